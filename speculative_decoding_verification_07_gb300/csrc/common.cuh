// Internal helpers shared by the CUDA translation units of the verification
// library: the handle, the device error word, the Philox4x32-10 generator,
// order-preserving keys and bounded acquire/release waits.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

struct sv_handle {
  int device;
  int num_sms;
  int* d_err;  // device error word: 0 or the first sv_status a kernel reported
  // launch cache: co-resident clusters per (kernel, cluster size), filled on
  // first use so later calls (and stream capture) make no occupancy query
  static constexpr int kCache = 32;
  const void* occ_fn[kCache];
  int occ_c[kCache];
  size_t occ_smem[kCache];
  int occ_val[kCache];
  int occ_n;
  // layout of the last spec_verify on a workspace: (pointer, kernel, B, kmax,
  // V, dtypes, histograms).  A call with another layout clears the scratch
  // words first, so a workspace may be reused for any shape.
  const void* ws_last;
  int64_t ws_key[6];
};

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Device error word: the first failure wins; later ones are dropped.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Raise a kernel's dynamic shared-memory limit to at least `bytes`, once per
// (kernel, size), under a process-wide mutex.  The attribute is per function:
// it is only ever raised, so a launch sized for an earlier limit stays valid
// whatever other threads set meanwhile (occupancy follows each launch's own
// dynamic size).
sv_status sv_raise_dyn_smem(const void* fn, size_t bytes);

// ---------------------------------------------------------------------------
// Acquire / release accesses at GPU scope (row states written by one cluster
// and polled by others).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Relaxed GPU-scope accesses: coherent, but order nothing else.  Used for
// words that carry their whole message themselves (the row-state words).
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the key
// bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// U = (2 * (r >> 9) + 1) * 2^-24: 23 random bits, exact in fp32, in (0, 1).
__device__ __forceinline__ float uniform_from_bits(uint32_t r) {
  return __uint2float_rn(((r >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
}

// ---------------------------------------------------------------------------
// Fast MUFU transcendentals (base 2).  ex2: ~2 ulp, results below 2^-126
// flush to 0.  lg2: absolute error ~2^-22.6.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch (sm_90+).  A kernel launched with the
// programmatic-stream-serialization attribute may start while the kernel
// before it in the stream is still running: pdl_wait() blocks until that
// kernel has completed and its writes are visible (for a kernel launched
// without the attribute it returns at once), and pdl_trigger() lets the next
// kernel in the stream start early and wait in its own pdl_wait().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order-preserving unsigned key of an fp32 value (-0 maps like +0).
__device__ __forceinline__ uint32_t fkey(float v) {
  uint32_t u = __float_as_uint(v);
  if (v == 0.0f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of fkey for keys of finite values.
__device__ __forceinline__ float fkey_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace sv

// Host side: launch with the programmatic-stream-serialization attribute (the
// kernel must call pdl_wait() before it reads anything an earlier kernel in
// the stream may still write).
template <typename... KArgs, typename... Args>
static inline cudaError_t sv_launch_pdl(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                        cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

// Host-side helper: map a CUDA error to SV_ERR_CUDA.
#define SV_CUDA_TRY(expr)                      \
  do {                                         \
    if ((expr) != cudaSuccess) return SV_ERR_CUDA; \
  } while (0)
