// Instantiations of the verification kernel (one nvcc process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_f32_f32_logits() { return &verify_kernel<4, 4, false, 4>; }
KernelFn kernel_f32_f32_probs() { return &verify_kernel<4, 4, true, 4>; }
KernelFn kernel_f32_bf16_logits() { return &verify_kernel<4, 2, false, 4>; }
}  // namespace sv
