// Stream-ordered update of one adapter's entries in a table's device lookup arrays (csrc/table_entry.cu).
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kMaxEntryBlocks = 64;                 // experts per adapter the update carries at most

struct TableEntry {
    uint64_t a[kMaxEntryBlocks], b[kMaxEntryBlocks];   // the adapter's A blocks (E_A of them) and B blocks (E_B)
    int32_t index, E_A, E_B, rpad;
    float scale;
};

// Writes entry `e` into a_ptr / b_ptr / rpad / scale with one single-thread kernel on `s`: launches enqueued
// on `s` before it read the old entry, launches after it the new one.
cudaError_t launch_set_entry(const TableEntry &e, uint64_t *a_ptr, uint64_t *b_ptr, int32_t *rpad, float *scale,
                             cudaStream_t s);

}  // namespace lora
