// Instantiations of the verification kernel with the top-k filter (one nvcc
// process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_bf16_bf16_logits_topk() { return &verify_kernel<2, 2, false, true>; }
}  // namespace sv
