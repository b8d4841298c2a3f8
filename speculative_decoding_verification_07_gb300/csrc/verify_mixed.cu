// Instantiations of the verification kernel (one nvcc process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_bf16_f32_probs() { return &verify_kernel<2, 4, true, false>; }
KernelFn kernel_bf16_f32_logits() { return &verify_kernel<2, 4, false, false>; }
}  // namespace sv
