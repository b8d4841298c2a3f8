// Instantiations of the verification kernel with the top-k filter (one nvcc
// process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_f32_f32_logits_topk() { return &verify_kernel<4, 4, false, true>; }
KernelFn kernel_f32_f32_probs_topk() { return &verify_kernel<4, 4, true, true>; }
KernelFn kernel_f32_bf16_logits_topk() { return &verify_kernel<4, 2, false, true>; }
}  // namespace sv
