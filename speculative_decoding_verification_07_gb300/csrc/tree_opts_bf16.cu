// Instantiations of the token-tree verification kernel with the request options
// (EOS ids, output caps, repetition penalty) compiled in (one nvcc process per file).
#include "tree_kernel.cuh"

namespace sv {
TreeKernelFn tree_kernel_bf16_bf16_logits_opts() { return &tree_kernel<2, 2, false, true>; }
TreeKernelFn tree_kernel_bf16_f32_probs_opts() { return &tree_kernel<2, 4, true, true>; }
TreeKernelFn tree_kernel_bf16_f32_logits_opts() { return &tree_kernel<2, 4, false, true>; }
}  // namespace sv
