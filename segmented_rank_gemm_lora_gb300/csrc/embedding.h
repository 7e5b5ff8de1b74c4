// Embedding LoRA (csrc/embedding.cu): parameters and launch, for the host side of the C ABI.
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kEmbedThreads = 256;
constexpr int kEmbedRows = 32;          // tokens of one tile

struct EmbedParams {
    // weight table: A packed over K = the vocabulary size V, one slice of N = the embedding width
    const uint64_t *a_ptr, *b_ptr;      // [L] packed block addresses
    const int32_t *rpad;                // [L] stored rank
    const float *scale;                 // [L]
    int32_t L, V, n_slices;
    int32_t slice_n[kMaxSlices], slice_off[kMaxSlices], slice_tile_off[kMaxSlices];
    // segment table of the last build, the tokens' vocabulary ids
    const int32_t *header, *perm;
    const int4 *segments;
    const int32_t *vocab;
    __nv_bfloat16 *y;  int64_t ldy;
    uint32_t *err;
};

cudaError_t launch_embedding(const EmbedParams &p, dim3 grid, cudaStream_t s, bool pdl);

}  // namespace lora
