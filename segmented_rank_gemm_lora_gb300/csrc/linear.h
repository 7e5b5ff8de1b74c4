// The LoRA linear layer (csrc/linear.cu): parameters and launch, for the host side of the C ABI.
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kLinearThreads = 256;
constexpr int kLinearRows = 128;        // tokens of one tile (MMA M)
constexpr int kLinearCols = 256;        // output columns of one tile (MMA N of the base product)
constexpr int kLinearBCols = 128;       // output columns of one packed B tile (two per output tile)
constexpr int kLinearK = 64;            // K columns of one pipeline stage
constexpr int kLinearBTileBytes = 2 * 16384;  // the output tile's B tiles (stored rank 64 at most) after the stages
// stage bytes at A blocks of R rows at most: x [8][128][8] + W (256 rows x 128 B) + A [8][R][8], 1 KB aligned
inline int linear_stage_bytes(int R) { return ((kLinearRows + kLinearCols + R) * kLinearK * 2 + 1023) / 1024 * 1024; }
constexpr int kLinearMaxStages = 6;

struct LinearParams {
    CUtensorMap w_map;                  // W bf16 [N][K] (row stride ldw): box 64 columns x 256 rows, 128-byte swizzle
    CUtensorMap x_map;                  // x bf16 [max_M][K] (row stride ldx): box 64 columns x 128 rows; tiles whose 128
                                        // rows are one run of consecutive rows inside the last build's M load through it
    const __nv_bfloat16 *x;  int64_t ldx;
    __nv_bfloat16 *y;        int64_t ldy;
    // weight table (dense)
    const uint64_t *a_ptr, *b_ptr;      // [L] packed block addresses
    const int32_t *rpad;                // [L] stored rank
    const float *scale;                 // [L]
    int32_t L, K, n_a, n_slices;
    int32_t tiles;                      // 256-column output tiles over all slices
    int32_t slice_n[kMaxSlices], slice_off[kMaxSlices], slice_tile_off[kMaxSlices];   // (B tiles: 128 columns)
    int32_t slice_ctile_off[kMaxSlices];   // first 256-column output tile of each slice
    // segment table of the last build
    const int32_t *header, *perm;
    const int4 *segments;
    // pipeline
    int32_t stages, stage_bytes;        // stages of [x 16 KB | W 16 KB | A (max rows) x 64 x 2 B]
    uint32_t *err;
    uint64_t timeout_ns;
};

cudaError_t launch_linear(const LinearParams &p, dim3 grid, size_t smem, cudaStream_t s, bool pdl);
const void *linear_kernel_ptr();

}  // namespace lora
