// Instantiations of the token-tree verification kernel (one nvcc process per file).
#include "tree_kernel.cuh"

namespace sv {
TreeKernelFn tree_kernel_bf16_bf16_logits() { return &tree_kernel<2, 2, false, false>; }
TreeKernelFn tree_kernel_bf16_f32_probs() { return &tree_kernel<2, 4, true, false>; }
TreeKernelFn tree_kernel_bf16_f32_logits() { return &tree_kernel<2, 4, false, false>; }
}  // namespace sv
