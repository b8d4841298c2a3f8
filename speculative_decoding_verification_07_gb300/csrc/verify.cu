// Host entry of the batched verification step: argument checks, cluster
// sizing and the launch (see verify_kernel.cuh for the device design).
#include <cuda_runtime.h>
#include <stdint.h>

#include "verify_kernel.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Variant {
  KernelFn fn, fn_topk;
  int eb_t, eb_d;
  bool probs;
};

static const Variant kVariants[] = {
    // bf16 target, bf16 draft logits
    {kernel_bf16_bf16_logits(), kernel_bf16_bf16_logits_topk(), 2, 2, false},
    // bf16 target, fp32 draft probabilities
    {kernel_bf16_f32_probs(), kernel_bf16_f32_probs_topk(), 2, 4, true},
    // bf16 target, fp32 draft logits
    {kernel_bf16_f32_logits(), kernel_bf16_f32_logits_topk(), 2, 4, false},
    // fp32 target, fp32 draft logits
    {kernel_f32_f32_logits(), kernel_f32_f32_logits_topk(), 4, 4, false},
    // fp32 target, fp32 draft probabilities
    {kernel_f32_f32_probs(), kernel_f32_f32_probs_topk(), 4, 4, true},
    // fp32 target, bf16 draft logits
    {kernel_f32_bf16_logits(), kernel_f32_bf16_logits_topk(), 4, 2, false},
};

static int elem_bytes(int dt) { return dt == SV_BF16 ? 2 : 4; }

size_t workspace_bytes_for(int B, int kmax) {
  const size_t rows = (size_t)B * (size_t)(kmax + 1);
  return kHdrBytes + ((rows * 4 + 255) / 256) * 256;
}

// The streaming kernel (stream.cu) serves most calls; the cluster kernel
// above serves top-k, the repetition penalty and top-p on fp32 rows.
bool stream_eligible(const sv_verify_args* a);
size_t stream_workspace_bytes(const sv_verify_args* a);
size_t stream_state_bytes(const sv_verify_args* a);  // header + both state halves
sv_status stream_launch(sv_handle* h, const sv_verify_args* a, void* ws, size_t ws_bytes,
                        cudaStream_t stream);

}  // namespace sv

using namespace sv;

extern "C" size_t sv_verify_args_size(void) { return sizeof(sv_verify_args); }

extern "C" sv_status sv_workspace_size(const sv_verify_args* a, size_t* bytes) {
  if (!a || !bytes || a->B < 0 || a->kmax < 0) return SV_ERR_INVALID;
  const size_t cl = workspace_bytes_for(a->B, a->kmax);
  const size_t sb = stream_workspace_bytes(a);
  *bytes = sb > cl ? sb : cl;
  return SV_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

extern "C" sv_status spec_verify(sv_handle* h, const sv_verify_args* a, void* ws, size_t ws_bytes,
                                 sv_stream_t stream) {
  if (!h || !a) return SV_ERR_INVALID;
  if (a->B < 0 || a->kmax < 0 || a->kmax > kMaxK || a->V < 1) return SV_ERR_INVALID;
  if (a->B == 0) return SV_OK;
  if (a->target_dtype != SV_BF16 && a->target_dtype != SV_FP32) return SV_ERR_INVALID;
  if (a->draft_dtype != SV_BF16 && a->draft_dtype != SV_FP32) return SV_ERR_INVALID;
  if (a->draft_kind != SV_DRAFT_LOGITS && a->draft_kind != SV_DRAFT_PROBS) return SV_ERR_INVALID;
  if (a->draft_kind == SV_DRAFT_PROBS && a->draft_dtype != SV_FP32) return SV_ERR_UNSUPPORTED;
  const int ebt = elem_bytes(a->target_dtype), ebd = elem_bytes(a->draft_dtype);
  if (!a->target || !a->temperature || !a->accepted || !a->out_tokens || !a->num_emitted ||
      !a->status)
    return SV_ERR_INVALID;
  if (a->kmax > 0 && (!a->draft || !a->draft_tokens)) return SV_ERR_INVALID;
  if (a->rep_penalty && (a->rep_ld < 0 || a->rep_ld > kMaxRepLd || (a->rep_ld > 0 && !a->rep_tokens)))
    return SV_ERR_INVALID;
  if (a->target_ld < a->V || (a->target_ld * ebt) % 16 || !aligned16(a->target))
    return SV_ERR_INVALID;
  if (a->kmax > 0 && (a->draft_ld < a->V || (a->draft_ld * ebd) % 16 || !aligned16(a->draft)))
    return SV_ERR_INVALID;
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < workspace_bytes_for(a->B, a->kmax))
    return SV_ERR_INVALID;
  const size_t n_tickets = (size_t)a->B * (size_t)(a->kmax + 1);
  if (n_tickets > 0x7FFFFFFF) return SV_ERR_UNSUPPORTED;

  const bool use_stream = stream_eligible(a);
  {
    // The scratch words of both kernels sit at offsets that depend on the
    // call's shape: on a change of layout (or of workspace) clear them first.
    const int64_t key[6] = {use_stream ? 1 : 0, a->B, a->kmax, a->V,
                            (int64_t)a->target_dtype * 16 + a->draft_dtype * 4 + a->draft_kind,
                            a->top_p ? 1 : 0};
    bool same = h->ws_last == ws;
    for (int j = 0; j < 6 && same; ++j) same = h->ws_key[j] == key[j];
    if (!same) {
      size_t n = workspace_bytes_for(a->B, a->kmax);
      if (use_stream) {
        const size_t sb = stream_state_bytes(a);
        if (sb > n) n = sb;
      }
      if (n > ws_bytes) n = ws_bytes;
      SV_CUDA_TRY(cudaMemsetAsync(ws, 0, n, (cudaStream_t)stream));
      h->ws_last = ws;
      for (int j = 0; j < 6; ++j) h->ws_key[j] = key[j];
    }
  }
  if (use_stream) return stream_launch(h, a, ws, ws_bytes, (cudaStream_t)stream);

  const bool probs = a->draft_kind == SV_DRAFT_PROBS;
  const Variant* var = nullptr;
  for (const Variant& v : kVariants)
    if (v.eb_t == ebt && v.eb_d == ebd && v.probs == probs) var = &v;
  if (!var) return SV_ERR_UNSUPPORTED;
  const KernelFn fn = a->top_k ? var->fn_topk : var->fn;

  // Cluster size: the smallest whose slices fit kMaxBlk TMA blocks (any size,
  // not only powers of two: V = 151936 takes 10 CTAs rather than 16, so more
  // clusters are in flight), then doubled, up to 8, while the grid would leave
  // SMs idle.
  const int cap = kMaxBlk * kBlk;
  const size_t need = ((size_t)a->V + cap - 1) / cap;
  if (need > (size_t)kMaxCluster) return SV_ERR_UNSUPPORTED;
  int C = need < 1 ? 1 : (int)need;
  const size_t rows = n_tickets;
  while (2 * C <= 8 && rows * (size_t)C < (size_t)h->num_sms * 2) C <<= 1;
  int slice = (int)(((size_t)a->V + C - 1) / C);
  slice = (slice + kGroup - 1) / kGroup * kGroup;
  const int d_off = (slice * ebt + 127) / 128 * 128;
  const size_t dyn = (size_t)d_off + (size_t)slice * ebd;

  KParams P;
  P.B = a->B, P.kmax = a->kmax, P.V = a->V, P.flags = a->flags;
  P.target = (const char*)a->target, P.t_ld = a->target_ld;
  P.draft = (const char*)a->draft, P.d_ld = a->draft_ld;
  P.tokens = a->draft_tokens, P.k = a->k, P.temperature = a->temperature, P.top_p = a->top_p;
  P.request_id = a->request_id, P.seq_len = a->seq_len;
  P.seed_lo = (uint32_t)(a->seed & 0xFFFFFFFFu), P.seed_hi = (uint32_t)(a->seed >> 32);
  P.accepted = a->accepted, P.out_tokens = a->out_tokens, P.num_emitted = a->num_emitted;
  P.status = a->status, P.debug = a->debug, P.probs_p = a->probs_p, P.probs_q = a->probs_q;
  P.hdr = (uint32_t*)ws;
  P.row_state = (uint32_t*)((char*)ws + kHdrBytes);
  P.err = h->d_err;
  P.slice = slice, P.d_off = d_off, P.n_tickets = (int)n_tickets;
  P.spin_limit = (a->flags & SV_FLAG_TEST_WITHHOLD) ? 1024 : kDefaultSpin;
  P.eos = a->eos_id, P.max_new = a->max_new;
  P.top_k = a->top_k;
  P.rep_penalty = a->rep_penalty, P.rep_tokens = a->rep_tokens;
  P.rep_ld = a->rep_penalty ? (int)a->rep_ld : 0;
  P.rep_draft = a->draft_kind == SV_DRAFT_LOGITS;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = (cudaStream_t)stream;
  int max_clusters = 0;
  for (int i = 0; i < h->occ_n; ++i)
    if (h->occ_fn[i] == (const void*)fn && h->occ_c[i] == C && h->occ_smem[i] == dyn)
      max_clusters = h->occ_val[i];
  {
    const sv_status rs = sv_raise_dyn_smem((const void*)fn, dyn);
    if (rs != SV_OK) return rs;
  }
  if (max_clusters == 0) {
    if (C > 8)
      SV_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    cfg.gridDim = dim3((unsigned)C);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess ||
        max_clusters < 1) {
      (void)cudaGetLastError();
      return SV_ERR_UNSUPPORTED;
    }
    if (h->occ_n < sv_handle::kCache) {
      h->occ_fn[h->occ_n] = (const void*)fn;
      h->occ_c[h->occ_n] = C;
      h->occ_smem[h->occ_n] = dyn;
      h->occ_val[h->occ_n] = max_clusters;
      ++h->occ_n;
    }
  }
  const size_t nclusters = rows < (size_t)max_clusters ? rows : (size_t)max_clusters;
  cfg.gridDim = dim3((unsigned)(nclusters * C));
  // programmatic dependent launch: the kernel waits for its predecessor in
  // its first instruction (griddepcontrol.wait), so only its launch overlaps
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, fn, P) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return SV_OK;
}
