// Instantiations of the verification kernel with the top-k filter (one nvcc
// process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_bf16_f32_probs_topk() { return &verify_kernel<2, 4, true, true>; }
KernelFn kernel_bf16_f32_logits_topk() { return &verify_kernel<2, 4, false, true>; }
}  // namespace sv
