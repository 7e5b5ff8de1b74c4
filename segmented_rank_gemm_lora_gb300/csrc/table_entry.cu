// One adapter's table entries rewritten on the stream, for hot-swapping an
// adapter in a live table ("vLLM-Ascend dynamic LoRA fused operator", section
// 4.3: replacing an adapter while steps run needs a version lock or a double
// buffer; here the new weights go to a free pool block and only the lookup
// entries change, in stream order, so a step reads either the old adapter or
// the new one, never a mix).
#include "table_entry.h"

namespace lora {

__global__ void set_entry_kernel(const TableEntry e, uint64_t *a_ptr, uint64_t *b_ptr, int32_t *rpad, float *scale)
{
    for (int i = 0; i < e.E_A; ++i) a_ptr[(int64_t)e.index * e.E_A + i] = e.a[i];
    for (int i = 0; i < e.E_B; ++i) b_ptr[(int64_t)e.index * e.E_B + i] = e.b[i];
    rpad[e.index] = e.rpad;
    scale[e.index] = e.scale;
}

cudaError_t launch_set_entry(const TableEntry &e, uint64_t *a_ptr, uint64_t *b_ptr, int32_t *rpad, float *scale,
                             cudaStream_t s)
{
    set_entry_kernel<<<1, 1, 0, s>>>(e, a_ptr, b_ptr, rpad, scale);
    return cudaGetLastError();
}

}  // namespace lora
