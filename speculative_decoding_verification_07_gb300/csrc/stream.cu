// Host side of the streaming verification kernel (stream_kernel.cuh): which
// calls it serves, the workspace layout, and the launch.  Also instantiates
// the bf16 target / bf16 draft-logit variant (the other dtype mixes are in
// stream_more.cu).
#include <cuda_runtime.h>
#include <stdint.h>

#include "stream_body.cuh"

namespace sv {

StreamFn stream_bf16_bf16_logits() { return stream::stream_kernel<2, 2, false>; }

namespace {

using ProbsFn = void (*)(stream::SParams, float*, float*);

struct SVariant {
  StreamFn (*fn)();
  ProbsFn probs;
  int eb_t, eb_d;
  bool probs_kind;
  int chunk, dyn_smem;
};

template <int EBT, int EBD, bool PROBS>
constexpr int dyn_bytes() {
  return stream::num_stages<EBT, EBD>() * stream::stage_bytes<EBT, EBD>();
}

}  // namespace

ProbsFn probs_fn_bf16_bf16_logits() { return stream::stream_probs_kernel<2, 2, false>; }
ProbsFn probs_fn_bf16_f32_probs();
ProbsFn probs_fn_bf16_f32_logits();
ProbsFn probs_fn_f32_f32_logits();
ProbsFn probs_fn_f32_f32_probs();
ProbsFn probs_fn_f32_bf16_logits();

namespace {

const SVariant kStreamVariants[] = {
    {stream_bf16_bf16_logits, probs_fn_bf16_bf16_logits(), 2, 2, false,
     stream::chunk_elems<2, 2>(), dyn_bytes<2, 2, false>()},
    {stream_bf16_f32_probs, probs_fn_bf16_f32_probs(), 2, 4, true, stream::chunk_elems<2, 4>(),
     dyn_bytes<2, 4, true>()},
    {stream_bf16_f32_logits, probs_fn_bf16_f32_logits(), 2, 4, false, stream::chunk_elems<2, 4>(),
     dyn_bytes<2, 4, false>()},
    {stream_f32_f32_logits, probs_fn_f32_f32_logits(), 4, 4, false, stream::chunk_elems<4, 4>(),
     dyn_bytes<4, 4, false>()},
    {stream_f32_f32_probs, probs_fn_f32_f32_probs(), 4, 4, true, stream::chunk_elems<4, 4>(),
     dyn_bytes<4, 4, true>()},
    {stream_f32_bf16_logits, probs_fn_f32_bf16_logits(), 4, 2, false, stream::chunk_elems<4, 2>(),
     dyn_bytes<4, 2, false>()},
};

int eb_of(int dt) { return dt == SV_BF16 ? 2 : 4; }

const SVariant* find_variant(const sv_verify_args* a) {
  const int ebt = eb_of(a->target_dtype), ebd = eb_of(a->draft_dtype);
  const bool probs = a->draft_kind == SV_DRAFT_PROBS;
  for (const SVariant& v : kStreamVariants)
    if (v.eb_t == ebt && v.eb_d == ebd && v.probs_kind == probs) return &v;
  return nullptr;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct Layout {
  size_t state0, state1, state_bytes, rows, pstats, parts, total;
  int n_ch, part_bytes, hist;
};

Layout layout_for(const sv_verify_args* a, const SVariant& v) {
  Layout L;
  L.n_ch = (a->V + v.chunk - 1) / v.chunk;
  L.hist = (a->top_p != nullptr && v.eb_t == 2 && v.eb_d == 2 && !v.probs_kind) ? 1 : 0;
  L.part_bytes = stream::kPartHead + (L.hist ? 2 * 512 : 0);  // 16-byte aligned
  const size_t pairs = (size_t)a->B * (size_t)(a->kmax + 1);
  L.state_bytes = align256(stream::state_bytes_for(a->B, a->kmax));
  L.state0 = align256(workspace_bytes_for(a->B, a->kmax));
  L.state1 = L.state0 + L.state_bytes;
  L.rows = L.state1 + L.state_bytes;
  L.pstats = L.rows + align256(pairs * sizeof(stream::RowRec));
  L.parts = L.pstats + align256(pairs * sizeof(stream::PairStats));
  L.total = L.parts + align256(pairs * (size_t)L.n_ch * (size_t)L.part_bytes);
  return L;
}

}  // namespace

// Calls the streaming kernel serves (when SV_FLAG_STREAM_PATH asks for it): no
// top-k, no repetition penalty, V within 32 chunks, and top-p only on bf16
// logit rows (fp32 rows with top-p, and the other options, go to the cluster
// kernel).  fp32 rows need ld % 8 == 0 so that whole 8-element groups stay
// inside each row.
bool stream_eligible(const sv_verify_args* a) {
  if (!(a->flags & SV_FLAG_STREAM_PATH) || (a->flags & SV_FLAG_CLUSTER_PATH)) return false;
  if (a->top_k || a->rep_penalty) return false;
  const SVariant* v = find_variant(a);
  if (!v) return false;
  if ((size_t)a->V > (size_t)stream::kMaxChunks * (size_t)v->chunk) return false;
  const bool bf16_logits = v->eb_t == 2 && v->eb_d == 2 && !v->probs_kind;
  if (a->top_p && !bf16_logits) return false;
  if (v->eb_t == 4 && (a->target_ld % 8) != 0) return false;
  if (a->kmax > 0 && v->eb_d == 4 && (a->draft_ld % 8) != 0) return false;
  return true;
}

size_t stream_workspace_bytes(const sv_verify_args* a) {
  const SVariant* v = find_variant(a);
  if (!v || a->B < 0 || a->kmax < 0 || a->V < 1) return 0;
  return layout_for(a, *v).total;
}

size_t stream_state_bytes(const sv_verify_args* a) {
  const SVariant* v = find_variant(a);
  if (!v || a->B < 0 || a->kmax < 0 || a->V < 1) return 0;
  return layout_for(a, *v).rows;
}

sv_status stream_launch(sv_handle* h, const sv_verify_args* a, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  const SVariant* v = find_variant(a);
  if (!v) return SV_ERR_UNSUPPORTED;
  const Layout L = layout_for(a, *v);
  if (ws_bytes < L.total) return SV_ERR_INVALID;
  const size_t pairs = (size_t)a->B * (size_t)(a->kmax + 1);
  const int n_blk = (L.n_ch + stream::kBatch - 1) / stream::kBatch;
  const size_t n_static = pairs * (size_t)n_blk;
  const size_t n_slots = stream::slots_for(a->B, a->kmax);
  if (n_static + 4096 > 0xFFFFFFF0u || (n_slots + 1) * (size_t)L.n_ch + 4096 > 0xFFFFFFF0u)
    return SV_ERR_UNSUPPORTED;

  char* base = (char*)ws;
  stream::SParams P;
  P.B = a->B, P.kmax = a->kmax, P.V = a->V, P.n_ch = L.n_ch;
  P.flags = a->flags;
  P.target = (const char*)a->target, P.t_ld = a->target_ld;
  P.draft = (const char*)a->draft, P.d_ld = a->draft_ld;
  P.tokens = a->draft_tokens, P.k = a->k, P.temperature = a->temperature, P.top_p = a->top_p;
  P.request_id = a->request_id, P.seq_len = a->seq_len;
  P.seed_lo = (uint32_t)(a->seed & 0xFFFFFFFFu), P.seed_hi = (uint32_t)(a->seed >> 32);
  P.accepted = a->accepted, P.out_tokens = a->out_tokens, P.num_emitted = a->num_emitted;
  P.status = a->status, P.debug = a->debug;
  P.eos = a->eos_id, P.max_new = a->max_new;
  P.hdr = reinterpret_cast<stream::Hdr*>(base + 64);
  P.state[0] = base + L.state0;
  P.state[1] = base + L.state1;
  P.state_words = L.state_bytes / 4;
  P.rows = reinterpret_cast<stream::RowRec*>(base + L.rows);
  P.pstats = reinterpret_cast<stream::PairStats*>(base + L.pstats);
  P.parts = base + L.parts;
  P.n_slots = (uint32_t)n_slots;
  P.part_bytes = L.part_bytes;
  P.hist = L.hist;
  P.err = h->d_err;
  P.slot_wait_ns = (a->flags & SV_FLAG_TEST_WITHHOLD) ? 250000ull : 2000000000ull;
  P.n_static = (uint32_t)n_static;
  P.n_blk = n_blk;

  const StreamFn fn = v->fn();
  {
    const sv_status rs = sv_raise_dyn_smem((const void*)fn, (size_t)v->dyn_smem);
    if (rs != SV_OK) return rs;
  }
  if (sv_launch_pdl(fn, dim3((unsigned)h->num_sms), dim3(stream::kAllThreads), (size_t)v->dyn_smem,
                    stream, P) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  if (a->probs_p) {
    const dim3 grid((unsigned)pairs, (unsigned)L.n_ch);
    v->probs<<<grid, 256, 0, stream>>>(P, a->probs_p, a->kmax > 0 ? a->probs_q : nullptr);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace sv

#ifdef SV_TRACE
// Trace set-up of the instrumented build: `buf` holds grid x `cap` events of
// two 64-bit words (CTA c writes events [c * cap, (c + 1) * cap)).
extern "C" sv_status sv_trace_setup(void* buf, unsigned cap) {
  unsigned long long* p = (unsigned long long*)buf;
  const unsigned zero = 0u;
  SV_CUDA_TRY(cudaMemcpyToSymbol(sv::stream::g_sv_trace, &p, sizeof(p)));
  SV_CUDA_TRY(cudaMemcpyToSymbol(sv::stream::g_sv_trace_cap, &cap, sizeof(cap)));
  SV_CUDA_TRY(cudaMemcpyToSymbol(sv::stream::g_sv_trace_n, &zero, sizeof(zero)));
  return SV_OK;
}
#endif
