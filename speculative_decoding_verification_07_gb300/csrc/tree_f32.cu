// Instantiations of the token-tree verification kernel (one nvcc process per file).
#include "tree_kernel.cuh"

namespace sv {
TreeKernelFn tree_kernel_f32_f32_logits() { return &tree_kernel<4, 4, false, false>; }
TreeKernelFn tree_kernel_f32_f32_probs() { return &tree_kernel<4, 4, true, false>; }
TreeKernelFn tree_kernel_f32_bf16_logits() { return &tree_kernel<4, 2, false, false>; }
}  // namespace sv
