// Handle management and device error reporting for the verification library.
#include <cuda_runtime.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"

extern "C" sv_status sv_create(int device, sv_handle** out) {
  if (!out) return SV_ERR_INVALID;
  *out = nullptr;
  SV_CUDA_TRY(cudaSetDevice(device));
  int sms = 0;
  SV_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
  sv_handle* h = (sv_handle*)calloc(1, sizeof(sv_handle));
  if (!h) return SV_ERR_INVALID;
  h->device = device;
  h->num_sms = sms;
  if (cudaMalloc(&h->d_err, 256) != cudaSuccess || cudaMemset(h->d_err, 0, 256) != cudaSuccess) {
    free(h);
    return SV_ERR_CUDA;
  }
  *out = h;
  return SV_OK;
}

extern "C" sv_status sv_destroy(sv_handle* h) {
  if (!h) return SV_ERR_INVALID;
  const cudaError_t e = cudaFree(h->d_err);
  free(h);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status sv_get_error(sv_handle* h, sv_stream_t stream, int32_t* code) {
  if (!h || !code) return SV_ERR_INVALID;
  SV_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  int v = 0;
  SV_CUDA_TRY(cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  SV_CUDA_TRY(cudaMemset(h->d_err, 0, sizeof(int)));
  *code = v;
  return SV_OK;
}

namespace {
std::mutex g_smem_mu;
const void* g_smem_fn[64];
size_t g_smem_bytes[64];
int g_smem_n = 0;
}  // namespace

sv_status sv::sv_raise_dyn_smem(const void* fn, size_t bytes) {
  std::lock_guard<std::mutex> lock(g_smem_mu);
  int i = 0;
  while (i < g_smem_n && g_smem_fn[i] != fn) ++i;
  if (i < g_smem_n && g_smem_bytes[i] >= bytes) return SV_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  if (i == g_smem_n) {
    if (g_smem_n == 64) return SV_OK;  // not recorded: the next call sets it again
    g_smem_fn[g_smem_n++] = fn;
  }
  g_smem_bytes[i] = bytes;
  return SV_OK;
}
