// Host entry of token-tree verification: argument checks, cluster sizing and
// the launch (see tree_kernel.cuh for the device design).
#include <cuda_runtime.h>
#include <stdint.h>

#include "tree_kernel.cuh"

using namespace sv;

namespace {

struct TreeVariant {
  TreeKernelFn fn, fn_opts;  // without / with the request options compiled in
  int eb_t, eb_d;
  bool probs;
};

const TreeVariant kTreeVariants[] = {
    {tree_kernel_bf16_bf16_logits(), tree_kernel_bf16_bf16_logits_opts(), 2, 2, false},
    {tree_kernel_bf16_f32_probs(), tree_kernel_bf16_f32_probs_opts(), 2, 4, true},
    {tree_kernel_bf16_f32_logits(), tree_kernel_bf16_f32_logits_opts(), 2, 4, false},
    {tree_kernel_f32_f32_logits(), tree_kernel_f32_f32_logits_opts(), 4, 4, false},
    {tree_kernel_f32_f32_probs(), tree_kernel_f32_f32_probs_opts(), 4, 4, true},
    {tree_kernel_f32_bf16_logits(), tree_kernel_f32_bf16_logits_opts(), 4, 2, false},
};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" size_t sv_tree_args_size(void) { return sizeof(sv_tree_args); }

extern "C" sv_status spec_verify_tree(sv_handle* h, const sv_tree_args* a, sv_stream_t stream) {
  if (!h || !a) return SV_ERR_INVALID;
  if (a->B < 0 || a->N < 0 || a->N > SV_TREE_MAX_NODES || a->V < 1) return SV_ERR_INVALID;
  if (a->B == 0) return SV_OK;
  if (a->target_dtype != SV_BF16 && a->target_dtype != SV_FP32) return SV_ERR_INVALID;
  if (a->draft_dtype != SV_BF16 && a->draft_dtype != SV_FP32) return SV_ERR_INVALID;
  if (a->draft_kind != SV_DRAFT_LOGITS && a->draft_kind != SV_DRAFT_PROBS) return SV_ERR_INVALID;
  if (a->draft_kind == SV_DRAFT_PROBS && a->draft_dtype != SV_FP32) return SV_ERR_UNSUPPORTED;
  const int ebt = a->target_dtype == SV_BF16 ? 2 : 4, ebd = a->draft_dtype == SV_BF16 ? 2 : 4;
  if (!a->target || !a->draft || !a->temperature || !a->accepted || !a->path || !a->out_tokens ||
      !a->num_emitted || !a->status)
    return SV_ERR_INVALID;
  if (a->N > 0 && (!a->parent || !a->tokens)) return SV_ERR_INVALID;
  if (a->rep_penalty && (a->rep_ld < 0 || a->rep_ld > kMaxRepLd || (a->rep_ld > 0 && !a->rep_tokens)))
    return SV_ERR_INVALID;
  if (a->target_ld < a->V || (a->target_ld * ebt) % 16 || !aligned16(a->target)) return SV_ERR_INVALID;
  if (a->draft_ld < a->V || (a->draft_ld * ebd) % 16 || !aligned16(a->draft)) return SV_ERR_INVALID;

  const bool probs = a->draft_kind == SV_DRAFT_PROBS;
  const TreeVariant* var = nullptr;
  for (const TreeVariant& v : kTreeVariants)
    if (v.eb_t == ebt && v.eb_d == ebd && v.probs == probs) var = &v;
  if (!var) return SV_ERR_UNSUPPORTED;

  // Cluster size as for the linear kernel: slices of at most kMaxBlk TMA
  // blocks, grown while the requests would leave SMs idle.
  const int cap = kMaxBlk * kBlk;
  int C = 1;
  while (C < kMaxCluster && (size_t)C * cap < (size_t)a->V) C <<= 1;
  if ((size_t)C * cap < (size_t)a->V) return SV_ERR_UNSUPPORTED;
  while (C < 8 && (size_t)a->B * C < (size_t)h->num_sms * 2) C <<= 1;
  int slice = (int)(((size_t)a->V + C - 1) / C);
  slice = (slice + kGroup - 1) / kGroup * kGroup;
  const int d_off = (slice * ebt + 127) / 128 * 128;
  const size_t dyn = (size_t)d_off + (size_t)slice * ebd;

  TreeParams P;
  P.B = a->B, P.N = a->N, P.V = a->V;
  P.target = (const char*)a->target, P.t_ld = a->target_ld;
  P.draft = (const char*)a->draft, P.d_ld = a->draft_ld;
  P.parent = a->parent, P.tokens = a->tokens, P.n_nodes = a->n_nodes;
  P.temperature = a->temperature, P.top_p = a->top_p, P.top_k = a->top_k;
  P.request_id = a->request_id, P.seq_len = a->seq_len;
  P.seed_lo = (uint32_t)(a->seed & 0xFFFFFFFFu), P.seed_hi = (uint32_t)(a->seed >> 32);
  P.accepted = a->accepted, P.path = a->path, P.out_tokens = a->out_tokens;
  P.num_emitted = a->num_emitted, P.status = a->status;
  P.eos = a->eos_id, P.max_new = a->max_new;
  P.rep_penalty = a->rep_penalty, P.rep_tokens = a->rep_tokens;
  P.rep_ld = a->rep_penalty ? (int)a->rep_ld : 0;
  P.rep_draft = a->draft_kind == SV_DRAFT_LOGITS;
  P.err = h->d_err;
  // the handle's 256 device bytes hold the error word at offset 0 and, at
  // offset 128, the request ticket and done counters (zero between calls)
  P.ctr = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(h->d_err) + 128);
  P.slice = slice, P.d_off = d_off;

  const bool opts = a->eos_id || a->max_new || a->rep_penalty;
  const TreeKernelFn fn = opts ? var->fn_opts : var->fn;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
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
    if (C > 8) SV_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    cfg.gridDim = dim3((unsigned)C);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess || max_clusters < 1) {
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
  const int nclusters = a->B < max_clusters ? a->B : max_clusters;
  cfg.gridDim = dim3((unsigned)(nclusters * C));
  if (cudaLaunchKernelEx(&cfg, fn, P) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return SV_OK;
}
