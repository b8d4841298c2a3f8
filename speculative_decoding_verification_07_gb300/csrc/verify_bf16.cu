// Instantiations of the verification kernel (one nvcc process per file).
#include "verify_kernel.cuh"

namespace sv {
KernelFn kernel_bf16_bf16_logits() { return &verify_kernel<2, 2, false, false>; }
}  // namespace sv
