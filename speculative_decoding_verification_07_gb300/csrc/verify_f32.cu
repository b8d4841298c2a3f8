// Instantiations of the verification kernel (one nvcc process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_f32_f32_logits() { return &verify_kernel<4, 4, false, false>; }
KernelFn kernel_f32_f32_probs() { return &verify_kernel<4, 4, true, false>; }
KernelFn kernel_f32_bf16_logits() { return &verify_kernel<4, 2, false, false>; }
}  // namespace sv
