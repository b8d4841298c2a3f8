// Streaming verification kernel: the dtype mixes other than bf16 target with
// bf16 draft logits (see stream.cu).
#include "stream_body.cuh"

namespace sv {

using ProbsFn = void (*)(stream::SParams, float*, float*);

StreamFn stream_bf16_f32_probs() { return stream::stream_kernel<2, 4, true>; }
StreamFn stream_bf16_f32_logits() { return stream::stream_kernel<2, 4, false>; }
StreamFn stream_f32_f32_logits() { return stream::stream_kernel<4, 4, false>; }
StreamFn stream_f32_f32_probs() { return stream::stream_kernel<4, 4, true>; }
StreamFn stream_f32_bf16_logits() { return stream::stream_kernel<4, 2, false>; }

ProbsFn probs_fn_bf16_f32_probs() { return stream::stream_probs_kernel<2, 4, true>; }
ProbsFn probs_fn_bf16_f32_logits() { return stream::stream_probs_kernel<2, 4, false>; }
ProbsFn probs_fn_f32_f32_logits() { return stream::stream_probs_kernel<4, 4, false>; }
ProbsFn probs_fn_f32_f32_probs() { return stream::stream_probs_kernel<4, 4, true>; }
ProbsFn probs_fn_f32_bf16_logits() { return stream::stream_probs_kernel<4, 2, false>; }

}  // namespace sv
