// spec_verify_static: the verification step for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they verify: code
// running inside a memory pool or allocator hook that must not re-enter the
// allocator, runtimes that own all device memory up front and hand out no
// scratch, or service loops that forbid allocation after start-up.  They still
// own their inputs and outputs; this entry point takes its scratch (the row
// ticket counter and the per-row decision words) from a fixed array in device
// global memory instead of a caller workspace, and it allocates nothing.
//
// Limits and behaviour, as a user should know them:
//  * The array holds at most SV_STATIC_MAX_ROWS = 16384 rows (B * (kmax + 1));
//    larger batches are refused with SV_ERR_TOO_LARGE before anything is
//    launched or queued.
//  * Every GPU that loads this library keeps the array (about 64 KB) until the
//    process exits.
//  * All calls in the process share the one array per device.  Each call
//    clears the counters and its own rows' decision words (one
//    cudaMemsetAsync on its stream, at most 64 KB), so no word from an older
//    call can carry a matching epoch tag.  Two calls whose work
//    overlaps on the GPU (for example on two streams without ordering) race
//    on the array and give wrong results: order them on one stream.
//  * The first call on a device looks up the array's address with
//    cudaGetSymbolAddress (and queries the device), with that device current;
//    make that first call before any stream capture.
//  * There is no handle, so no device error word: conditions the device
//    detects are reported only through the per-request status bits.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "verify_kernel.cuh"

namespace {

constexpr int kStaticRows = SV_STATIC_MAX_ROWS;
constexpr size_t kStaticBytes = sv::kHdrBytes + (size_t)kStaticRows * 4;
constexpr int kMaxDevices = 64;

// The scratch: workspace header (epoch, ticket, done counters) and one
// decision word per row.  Zero at module load.
static __device__ __align__(256) unsigned char g_static_ws[kStaticBytes];

struct StaticDevice {
  int ready;
  void* ws;   // device address of g_static_ws on this device
  int num_sms;
  // co-resident clusters per (kernel, cluster size, shared memory)
  const void* occ_fn[16];
  int occ_c[16];
  size_t occ_smem[16];
  int occ_val[16];
  int occ_n;
};

StaticDevice g_dev[kMaxDevices];
std::mutex g_mu;  // guards g_dev (set-up and the occupancy cache)

sv_status setup_device(int dev, StaticDevice** out) {
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_UNSUPPORTED;
  StaticDevice& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return SV_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return SV_ERR_CUDA;
    }
    d.ws = p;
    d.num_sms = sms;
    d.occ_n = 0;
    d.ready = 1;
  }
  *out = &d;
  return SV_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

sv::KernelFn pick_kernel(int ebt, int ebd, bool probs, bool topk) {
  using namespace sv;
  if (ebt == 2 && ebd == 2 && !probs) return topk ? kernel_bf16_bf16_logits_topk() : kernel_bf16_bf16_logits();
  if (ebt == 2 && ebd == 4 && probs) return topk ? kernel_bf16_f32_probs_topk() : kernel_bf16_f32_probs();
  if (ebt == 2 && ebd == 4 && !probs) return topk ? kernel_bf16_f32_logits_topk() : kernel_bf16_f32_logits();
  if (ebt == 4 && ebd == 4 && !probs) return topk ? kernel_f32_f32_logits_topk() : kernel_f32_f32_logits();
  if (ebt == 4 && ebd == 4 && probs) return topk ? kernel_f32_f32_probs_topk() : kernel_f32_f32_probs();
  if (ebt == 4 && ebd == 2 && !probs) return topk ? kernel_f32_bf16_logits_topk() : kernel_f32_bf16_logits();
  return nullptr;
}

}  // namespace

extern "C" sv_status spec_verify_static(const sv_verify_args* a, sv_stream_t stream) {
  using namespace sv;
  if (!a) return SV_ERR_INVALID;
  if (a->B < 0 || a->kmax < 0 || a->kmax > kMaxK || a->V < 1) return SV_ERR_INVALID;
  if (a->B == 0) return SV_OK;
  const size_t rows = (size_t)a->B * (size_t)(a->kmax + 1);
  if (rows > (size_t)kStaticRows) return SV_ERR_TOO_LARGE;  // beyond the fixed scratch
  if (a->target_dtype != SV_BF16 && a->target_dtype != SV_FP32) return SV_ERR_INVALID;
  if (a->draft_dtype != SV_BF16 && a->draft_dtype != SV_FP32) return SV_ERR_INVALID;
  if (a->draft_kind != SV_DRAFT_LOGITS && a->draft_kind != SV_DRAFT_PROBS) return SV_ERR_INVALID;
  if (a->draft_kind == SV_DRAFT_PROBS && a->draft_dtype != SV_FP32) return SV_ERR_UNSUPPORTED;
  const int ebt = a->target_dtype == SV_BF16 ? 2 : 4, ebd = a->draft_dtype == SV_BF16 ? 2 : 4;
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
  const bool probs = a->draft_kind == SV_DRAFT_PROBS;
  const KernelFn fn = pick_kernel(ebt, ebd, probs, a->top_k != nullptr);
  if (!fn) return SV_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  StaticDevice* d = nullptr;
  const sv_status st = setup_device(dev, &d);
  if (st != SV_OK) return st;

  // cluster size and slice, as for spec_verify
  const int cap = kMaxBlk * kBlk;
  const size_t need = ((size_t)a->V + cap - 1) / cap;
  if (need > (size_t)kMaxCluster) return SV_ERR_UNSUPPORTED;
  int C = need < 1 ? 1 : (int)need;
  while (2 * C <= 8 && rows * (size_t)C < (size_t)d->num_sms * 2) C <<= 1;
  int slice = (int)(((size_t)a->V + C - 1) / C);
  slice = (slice + kGroup - 1) / kGroup * kGroup;
  const int d_off = (slice * ebt + 127) / 128 * 128;
  const size_t dyn = (size_t)d_off + (size_t)slice * ebd;

  KParams P;
  memset(&P, 0, sizeof(P));
  P.B = a->B, P.kmax = a->kmax, P.V = a->V, P.flags = a->flags;
  P.target = (const char*)a->target, P.t_ld = a->target_ld;
  P.draft = (const char*)a->draft, P.d_ld = a->draft_ld;
  P.tokens = a->draft_tokens, P.k = a->k, P.temperature = a->temperature, P.top_p = a->top_p;
  P.request_id = a->request_id, P.seq_len = a->seq_len;
  P.seed_lo = (uint32_t)(a->seed & 0xFFFFFFFFu), P.seed_hi = (uint32_t)(a->seed >> 32);
  P.accepted = a->accepted, P.out_tokens = a->out_tokens, P.num_emitted = a->num_emitted;
  P.status = a->status, P.debug = a->debug, P.probs_p = a->probs_p, P.probs_q = a->probs_q;
  P.hdr = (uint32_t*)d->ws;
  P.row_state = (uint32_t*)((char*)d->ws + kHdrBytes);
  P.err = nullptr;  // no handle: device conditions go to the status bits only
  P.slice = slice, P.d_off = d_off, P.n_tickets = (int)rows;
  P.spin_limit = (a->flags & SV_FLAG_TEST_WITHHOLD) ? 1024 : kDefaultSpin;
  P.eos = a->eos_id, P.max_new = a->max_new;
  P.top_k = a->top_k;
  P.rep_penalty = a->rep_penalty, P.rep_tokens = a->rep_tokens;
  P.rep_ld = a->rep_penalty ? (int)a->rep_ld : 0;
  P.rep_draft = a->draft_kind == SV_DRAFT_LOGITS;

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
  {
    const sv_status rs = sv_raise_dyn_smem((const void*)fn, dyn);
    if (rs != SV_OK) return rs;
  }
  int max_clusters = 0;
  for (int i = 0; i < d->occ_n; ++i)
    if (d->occ_fn[i] == (const void*)fn && d->occ_c[i] == C && d->occ_smem[i] == dyn)
      max_clusters = d->occ_val[i];
  if (max_clusters == 0) {
    if (C > 8 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      (void)cudaGetLastError();
      return SV_ERR_CUDA;
    }
    cfg.gridDim = dim3((unsigned)C);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess || max_clusters < 1) {
      (void)cudaGetLastError();
      return SV_ERR_UNSUPPORTED;
    }
    if (d->occ_n < 16) {
      d->occ_fn[d->occ_n] = (const void*)fn;
      d->occ_c[d->occ_n] = C;
      d->occ_smem[d->occ_n] = dyn;
      d->occ_val[d->occ_n] = max_clusters;
      ++d->occ_n;
    }
  }
  // the ticket and done counters must start at zero, and so must this call's
  // row words (the epoch word stays): a word left from a call 2^28 epochs ago
  // would otherwise carry a matching tag
  if (cudaMemsetAsync((char*)d->ws + 4, 0, kHdrBytes - 4 + rows * 4, (cudaStream_t)stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  const size_t nclusters = rows < (size_t)max_clusters ? rows : (size_t)max_clusters;
  cfg.gridDim = dim3((unsigned)(nclusters * C));
  if (cudaLaunchKernelEx(&cfg, fn, P) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return SV_OK;
}
