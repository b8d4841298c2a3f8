#pragma once
// Batched verification step of speculative decoding on sm_103a (device code).
//
// Method ("Speculative decoding: accelerate LLM generation without changing
// its answers", sections 2-4): for each request b and draft position i, the
// temperature / top-p transformed target p_i and draft q_i; accept y_i iff
// u_i q_i(y_i) < p_i(y_i) (== u_i < min(1, p_i/q_i)), left to right; stop at
// the first rejection and draw the correction from normalize(max(0, p_i - q_i)),
// or the bonus token from p_{k_b} when every draft is accepted.  Both draws are
// exponential races argmax_x w_x / E_x with E_x = -ln U_x from Philox4x32-10.
//
// GB300 design
//  * One thread-block cluster of C CTAs owns one (request, position) row pair:
//    the target row and, for i < k_b, the draft row.  Each CTA streams its
//    1/C vocabulary slice once from HBM with 128-bit coalesced loads straight
//    into registers and keeps it there, so every later sweep (top-p histogram,
//    accept test, race) runs on-chip.  Row statistics are combined through
//    distributed shared memory (DSMEM) across the cluster.
//  * Single-sweep statistics: an online (max, sum of 2^((v-m)c)) per thread,
//    combined by rescaling; greedy rows (T = 0) count tied maxima instead.
//  * Top-p: a 256-bin histogram over the order-key distance from the row
//    maximum; for bf16 rows the first window is exact (one bin per bf16 value,
//    integer counts, deterministic).  Wider ranges descend radix-wise.
//  * Rows are handed out by a ticket counter in (position, request) order, so
//    a row only ever waits on rows with earlier tickets, which are already
//    held by running clusters (no deadlock); every wait is bounded.  A row
//    whose request already has a known earlier rejection is skipped without
//    being loaded.  Exactly one row per request -- the first rejection, or the
//    bonus row -- runs the race, and writes the request's outputs.
//  * The race prunes 4-token Philox groups that cannot beat the running best
//    (w / E_min below it) and evaluates an accurate logf only for candidates
//    the fast MUFU estimate cannot rule out.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = 8;               // elements per register group (one 16-byte bf16 vector)
constexpr uint32_t kNoFilter = 0xFFFFFFFFu;
constexpr int kMaxCluster = 16;
constexpr int kMaxK = 64;
constexpr int kDefaultSpin = 1 << 20;

// workspace header words
constexpr int kHdrEpoch = 0, kHdrTicket = 1, kHdrDone = 2;
constexpr size_t kHdrBytes = 256;

// row state word: (epoch << 4) | qzero << 3 | state
constexpr uint32_t kStateMask = 7u, kQZeroBit = 8u;

struct KParams {
  int B, kmax, V;
  uint32_t flags;
  const char* target;
  int64_t t_ld;  // elements
  const char* draft;
  int64_t d_ld;
  const int32_t* tokens;
  const int32_t* k;
  const float* temperature;
  const float* top_p;
  const uint32_t* request_id;
  const int32_t* seq_len;
  uint32_t seed_lo, seed_hi;
  int32_t* accepted;
  int32_t* out_tokens;
  int32_t* num_emitted;
  uint32_t* status;
  sv_row_debug* debug;
  float* probs_p;
  float* probs_q;
  uint32_t* hdr;
  uint32_t* row_state;
  int* err;
  int slice;      // elements per CTA (multiple of 8)
  int ng;         // register groups per thread in use (<= NG)
  int n_tickets;  // (kmax + 1) * B
  int spin_limit;
};

// ---------------------------------------------------------------------------
// Register groups of 8 elements: 4 words of bf16 pairs or 8 fp32 words.
// ---------------------------------------------------------------------------
template <int EB>
struct Grp {
  uint32_t w[EB * 2];
};

template <int EB>
__device__ __forceinline__ float gval(const Grp<EB>& g, int e) {
  if constexpr (EB == 2) {
    const uint32_t x = g.w[e >> 1];
    return __uint_as_float((e & 1) ? (x & 0xFFFF0000u) : (x << 16));
  } else {
    return __uint_as_float(g.w[e]);
  }
}

// Key used for top-p distances: bf16 rows use the 16-bit bf16 order key,
// fp32 rows the 32-bit one.
template <int EB>
__device__ __forceinline__ uint32_t vkey(float v) {
  return EB == 2 ? (fkey(v) >> 16) : fkey(v);
}

template <int EB>
__device__ __forceinline__ float vkey_value(uint32_t k) {
  if constexpr (EB == 2) {
    return fkey_value((k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu));
  } else {
    return fkey_value(k);
  }
}

// Streaming 16-byte load (read once; do not keep in L1).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Load one group of 8 elements starting at absolute element x of a row; lanes
// at or beyond `end` get the neutral value (-inf logits / 0 probabilities).
template <int EB, bool PROBS>
__device__ __forceinline__ void load_group(Grp<EB>& g, const char* row, int x, int end) {
  const uint32_t neutral = PROBS ? 0u : (EB == 2 ? 0xFF80FF80u : 0xFF800000u);
#pragma unroll
  for (int j = 0; j < EB * 2; ++j) g.w[j] = neutral;
  if (x >= end) return;
  const char* p = row + (size_t)x * EB;
  uint4 a = ld_stream(p);
  g.w[0] = a.x, g.w[1] = a.y, g.w[2] = a.z, g.w[3] = a.w;
  if constexpr (EB == 4) {
    if (x + 4 < end) {
      uint4 b2 = ld_stream(p + 16);
      g.w[4] = b2.x, g.w[5] = b2.y, g.w[6] = b2.z, g.w[7] = b2.w;
    }
  }
  if (x + kGroup > end) {  // ragged tail of the row: neutralise lanes >= end
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      if (x + e >= end) {
        if constexpr (EB == 2) {
          const uint32_t n16 = PROBS ? 0u : 0xFF80u;
          uint32_t& w = g.w[e >> 1];
          w = (e & 1) ? ((w & 0x0000FFFFu) | (n16 << 16)) : ((w & 0xFFFF0000u) | n16);
        } else {
          g.w[e] = neutral;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Per-row transform parameters (identical in every CTA of the cluster).
// ---------------------------------------------------------------------------
struct RowP {
  float m;          // maximum raw value (logit, or probability)
  float mz;         // maximum in the weight domain (logit, or lg2(prob)/T)
  float c;          // weight scale: log2(e)/T for logits, 1 for probabilities
  float invT;       // 1/T (probabilities)
  bool greedy;      // T == 0
  float S;          // sum of weights over the row (T > 0) / tie count (T == 0)
  float Z;          // normaliser of the kept set
  float invZ;
  uint32_t kmax;    // vkey(m)
  uint32_t Dstar;   // kept iff vkey(m) - vkey(v) <= Dstar; kNoFilter = all
};

// Unnormalised weight of a value: 2^((z - mz) c), or [v == m] for T = 0.
template <bool PROBS>
__device__ __forceinline__ float weight(float v, const RowP& r) {
  if (r.greedy) return v == r.m ? 1.0f : 0.0f;
  const float z = PROBS ? lg2(v) * r.invT : v;
  return ex2((z - r.mz) * r.c);
}

template <int EB>
__device__ __forceinline__ bool kept(float v, const RowP& r) {
  if (r.greedy) return v == r.m;
  if (r.Dstar == kNoFilter) return true;
  return (r.kmax - vkey<EB>(v)) <= r.Dstar;
}

template <int EB, bool PROBS>
__device__ __forceinline__ float prob(float v, const RowP& r) {
  return kept<EB>(v, r) ? weight<PROBS>(v, r) * r.invZ : 0.0f;
}

// ---------------------------------------------------------------------------
// Shared memory: block-reduction scratch plus the per-CTA partials other CTAs
// of the cluster read through DSMEM (one slot per phase so no slot is
// rewritten while a peer may still read it).
// ---------------------------------------------------------------------------
struct RacePart {
  float w, E;
  int idx;
};

struct Smem {
  int bcast[2][4];             // [iteration parity] ticket, kind (rank 0 only)
  int decide[4];               // resolver decision (rank 0 only)
  float st_m[2], st_s[2];      // stats partials: target, draft
  float st_raw;                // raw maximum of the draft row
  int st_bad[2];
  uint32_t hist[2][2][256];    // [buffer][row][bin]: counts or float bits
  RacePart race[2];            // [slot]
  float scratch_f[kWarps][4];
  int scratch_i[kWarps][4];
  RacePart scratch_r[kWarps];
  int bin_pick;
};

enum : int { kDone = 0, kNone = 1, kWork = 2 };

__device__ __forceinline__ bool better(float w1, float E1, int i1, float w2, float E2, int i2) {
  const float a = w1 * E2, b = w2 * E1;
  return a > b || (a == b && i1 < i2);
}

__device__ __forceinline__ void warp_race(float& w, float& E, int& idx) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float w2 = __shfl_xor_sync(0xffffffffu, w, o);
    const float E2 = __shfl_xor_sync(0xffffffffu, E, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (better(w2, E2, i2, w, E, idx)) w = w2, E = E2, idx = i2;
  }
}

// Combine online (max, sum) pairs: S = Sa 2^((ma-m)c) + Sb 2^((mb-m)c).
__device__ __forceinline__ void combine_ms(float& m, float& s, float m2, float s2, float c) {
  if (m2 > m) {
    s = (m == -INFINITY ? 0.0f : s * ex2((m - m2) * c)) + s2;
    m = m2;
  } else if (m2 != -INFINITY) {
    s += s2 * ex2((m2 - m) * c);
  }
}

// Per-row request parameters (uniform across the cluster).
struct Req {
  int b, i, kb;
  bool has_d;
  float T, top_p;
  bool params_ok;
  int y;
  int pos;
  uint32_t rid;
};

__device__ __forceinline__ uint32_t epoch_tag(uint32_t epoch) { return (epoch & 0x0FFFFFFFu) << 4; }

// Row-0 style check used by the ticket dispenser: has any earlier row of b
// already been decided as not accepted?
static __device__ bool earlier_not_accepted(const KParams& P, int b, int i, uint32_t epoch) {
  const uint32_t* rs = P.row_state + (size_t)b * (P.kmax + 1);
  for (int j = 0; j < i; ++j) {
    const uint32_t w = ld_acquire(rs + j);
    if ((w & ~0xFu) == epoch_tag(epoch) && (w & kStateMask) != 0 &&
        (w & kStateMask) != SV_ROW_ACCEPTED)
      return true;
  }
  return false;
}

static __device__ void write_bad_outputs(const KParams& P, int b, uint32_t st) {
  P.accepted[b] = -1;
  P.num_emitted[b] = 0;
  P.status[b] = st;
  for (int j = 0; j <= P.kmax; ++j) P.out_tokens[(size_t)b * (P.kmax + 1) + j] = -1;
}

// Histogram level for top-p: every element whose distance D = kmax - key lies
// in [lo, lo + 256 << shift) adds its count (COUNT) or weight to bin
// (D - lo) >> shift.
template <int EB, bool PROBS, bool COUNT, int NG>
__device__ __forceinline__ void hist_level(const Grp<EB> (&g)[NG], int ng, const RowP& r,
                                           uint32_t lo, int shift, uint32_t* hist) {
  const uint32_t span = shift >= 24 ? 0xFFFFFFFFu : ((256u << shift) - 1u);
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    if (gi >= ng) break;
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      const float v = gval<EB>(g[gi], e);
      const uint32_t D = r.kmax - vkey<EB>(v);
      const uint32_t u = D - lo;
      if (D >= lo && u <= span && v > (PROBS ? 0.0f : -INFINITY)) {
        const uint32_t bin = u >> shift;
        if (COUNT) {
          atomicAdd(&hist[bin], 1u);
        } else {
          atomicAdd(reinterpret_cast<float*>(&hist[bin]), weight<PROBS>(v, r));
        }
      }
    }
  }
}

// Inclusive block scan of one float per thread (thread t holds bin t).
__device__ __forceinline__ float block_scan(float v, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sm.scratch_f[warp][0] = v;
  __syncthreads();
  float off = 0.0f;
  for (int w = 0; w < warp; ++w) off += sm.scratch_f[w][0];
  __syncthreads();
  return v + off;
}

// Top-p threshold of one or two rows (target and, if has_d, draft) held in
// registers across the cluster.  Sets r.Dstar and r.Z.  All control flow
// depends only on cluster-reduced values, so every CTA takes the same path.
template <int EBT, int EBD, bool PROBS, int NG>
__device__ void top_p_rows(cg::cluster_group& cluster, Smem& sm, const Grp<EBT> (&tg)[NG],
                           const Grp<EBD> (&dg)[NG], int ng, bool has_d, float top_p, RowP& rt,
                           RowP& rd) {
  const int C = cluster.num_blocks();
  const int tid = threadIdx.x;
  struct Lv {
    uint32_t lo;
    int shift;
    float above;
    bool window, done;
    float R;
  } L[2];
  L[0] = {0u, EBT == 2 ? 0 : 24, 0.0f, EBT == 2, false, top_p * rt.S};
  L[1] = {0u, EBD == 2 ? 0 : 24, 0.0f, EBD == 2, !has_d, top_p * rd.S};
  int buf = 0;
  while (!(L[0].done && L[1].done)) {
    // 1. local histograms
    for (int j = tid; j < 512; j += kThreads) (&sm.hist[buf][0][0])[j] = 0u;
    __syncthreads();
    if (!L[0].done) {
      if (L[0].window && EBT == 2)
        hist_level<EBT, false, true>(tg, ng, rt, L[0].lo, L[0].shift, sm.hist[buf][0]);
      else
        hist_level<EBT, false, false>(tg, ng, rt, L[0].lo, L[0].shift, sm.hist[buf][0]);
    }
    if (!L[1].done) {
      if (L[1].window && EBD == 2)
        hist_level<EBD, PROBS, true>(dg, ng, rd, L[1].lo, L[1].shift, sm.hist[buf][1]);
      else
        hist_level<EBD, PROBS, false>(dg, ng, rd, L[1].lo, L[1].shift, sm.hist[buf][1]);
    }
    __syncthreads();
    cluster.sync();
    // 2. cluster-reduce bin t in thread t, then scan and pick the boundary bin
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      Lv& lv = L[row];
      if (lv.done) continue;
      const RowP& r = row == 0 ? rt : rd;
      const bool count = row == 0 ? (lv.window && EBT == 2) : (lv.window && EBD == 2);
      float h = 0.0f;
      if (count) {
        uint32_t n = 0;
        for (int q = 0; q < C; ++q) n += cluster.map_shared_rank(&sm.hist[buf][row][0], q)[tid];
        if (n) {
          const float v = row == 0 ? vkey_value<EBT>(r.kmax - lv.lo - (uint32_t)tid)
                                   : vkey_value<EBD>(r.kmax - lv.lo - (uint32_t)tid);
          h = (float)n * (row == 0 ? weight<false>(v, r) : weight<PROBS>(v, r));
        }
      } else {
        for (int q = 0; q < C; ++q)
          h += __uint_as_float(cluster.map_shared_rank(&sm.hist[buf][row][0], q)[tid]);
      }
      const float incl = block_scan(h, sm);
      if (tid == 0) sm.bin_pick = 256;
      __syncthreads();
      const float excl = incl - h;
      if (lv.above + incl >= lv.R && lv.above + excl < lv.R) atomicMin(&sm.bin_pick, tid);
      __syncthreads();
      int c = sm.bin_pick;
      if (c == 256) {
        if (lv.window) {  // boundary lies beyond the exact window: full radix descent
          lv.window = false;
          lv.lo = 0u;
          lv.above = 0.0f;
          lv.shift = (row == 0 ? EBT : EBD) == 2 ? 8 : 24;
          __syncthreads();
          continue;
        }
        // rounding left the target mass unreachable: keep through the last non-empty bin
        if (tid == 0) sm.bin_pick = -1;
        __syncthreads();
        if (h > 0.0f) atomicMax(&sm.bin_pick, tid);
        __syncthreads();
        c = sm.bin_pick < 0 ? 0 : sm.bin_pick;
      }
      // broadcast the picked bin's exclusive prefix and mass from thread c
      if (tid == c) {
        sm.scratch_f[0][2] = excl;
        sm.scratch_f[0][3] = h;
      }
      __syncthreads();
      const float cexcl = sm.scratch_f[0][2], ch = sm.scratch_f[0][3];
      __syncthreads();
      lv.above += cexcl;
      lv.lo += (uint32_t)c << lv.shift;
      if (lv.shift == 0) {
        RowP& w = row == 0 ? rt : rd;
        w.Dstar = lv.lo;
        w.Z = lv.above + ch;
        w.invZ = 1.0f / w.Z;
        lv.done = true;
      } else {
        lv.shift -= 8;
      }
    }
    buf ^= 1;
  }
}

// Exponential race over the thread's register-resident slice.
//   bonus: w_x = kept p weight (unnormalised); residual: w_x = max(0, p_x - q_x).
template <int EBT, int EBD, bool PROBS, int NG>
__device__ __forceinline__ void race_slice(const Grp<EBT> (&tg)[NG], const Grp<EBD> (&dg)[NG],
                                           int ng, int x_base, bool residual, const RowP& rt,
                                           const RowP& rd, uint32_t pos, uint32_t rid,
                                           uint32_t k0, uint32_t k1, float& bw, float& bE,
                                           int& bidx) {
  // E >= E_min = -ln(1 - 2^-24) = 5.96e-8; a group whose largest w satisfies
  // w / E_min < best cannot win.
  constexpr float kEminSafe = 5.9604e-8f;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    if (gi >= ng) break;
    const int x = x_base + gi * kThreads * kGroup;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = h * 4 + j;
        const float vp = gval<EBT>(tg[gi], e);
        if (residual) {
          const float vq = gval<EBD>(dg[gi], e);
          w[j] = fmaxf(0.0f, prob<EBT, false>(vp, rt) - prob<EBD, PROBS>(vq, rd));
        } else {
          w[j] = kept<EBT>(vp, rt) ? weight<false>(vp, rt) : 0.0f;
        }
      }
      const float wm = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
      if (!(wm * bE > bw * kEminSafe)) continue;
      const int x4 = x + h * 4;
      const uint4 r = philox4x32_10(make_uint4((uint32_t)x4 >> 2, pos, rid, 0u), k0, k1);
      const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!(w[j] > 0.0f)) continue;
        const float U = uniform_from_bits(rr[j]);
        const float Ef = -lg2(U) * kLn2;
        const float Elo = Ef * (1.0f - 2e-6f) - 2e-7f;  // lower bound of the exact E
        if (Elo <= 0.0f || w[j] * bE > bw * Elo) {
          const float E = -logf(U);
          if (w[j] * bE > bw * E) bw = w[j], bE = E, bidx = x4 + j;
        }
      }
    }
  }
}

template <int EBT, int EBD, bool PROBS, int NG>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const KParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ Smem sm;
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t epoch = *(volatile const uint32_t*)(P.hdr + kHdrEpoch);
  const uint32_t tag = epoch_tag(epoch);
  const uint32_t k0 = P.seed_lo, k1 = P.seed_hi;

  // rank 0 hands out tickets in (position, request) order
  auto grab = [&](int parity) {
    if (rank == 0 && tid == 0) {
      int kind = kDone, t = 0;
      for (;;) {
        t = (int)atomicAdd(P.hdr + kHdrTicket, 1u);
        if (t >= P.n_tickets) { kind = kDone; break; }
        const int i = t / P.B, b = t - i * P.B;
        const int kb = P.k ? P.k[b] : P.kmax;
        if (kb < 0 || kb > P.kmax) {
          if (i == 0) write_bad_outputs(P, b, SV_ST_BAD_INPUT);
          continue;
        }
        if (i > kb) continue;
        if (!(P.flags & SV_FLAG_NO_SKIP) && earlier_not_accepted(P, b, i, epoch)) {
          st_release(P.row_state + (size_t)b * (P.kmax + 1) + i, tag | SV_ROW_SKIPPED);
          if (P.debug) P.debug[(size_t)b * (P.kmax + 1) + i].state = SV_ROW_SKIPPED;
          continue;
        }
        kind = kWork;
        break;
      }
      sm.bcast[parity][0] = t;
      sm.bcast[parity][1] = kind;
    }
  };

  grab(0);
  cluster.sync();
  for (int it = 0;; ++it) {
    const int parity = it & 1;
    const int* bc = cluster.map_shared_rank(&sm.bcast[parity][0], 0);
    const int t = bc[0], kind = bc[1];
    if (kind == kDone) break;

    // ---------------------------------------------------------------- row setup
    Req q;
    q.i = t / P.B;
    q.b = t - q.i * P.B;
    q.kb = P.k ? P.k[q.b] : P.kmax;
    q.has_d = q.i < q.kb;
    q.T = P.temperature[q.b];
    q.top_p = P.top_p ? P.top_p[q.b] : 1.0f;
    q.params_ok = (q.T >= 0.0f) && (q.T <= FLT_MAX) && (q.top_p > 0.0f) && (q.top_p <= 1.0f);
    q.y = q.has_d ? P.tokens[(size_t)q.b * P.kmax + q.i] : 0;
    q.pos = (P.seq_len ? P.seq_len[q.b] : 0) + 1 + q.i;
    q.rid = P.request_id ? P.request_id[q.b] : (uint32_t)q.b;
    const bool y_ok = !q.has_d || (q.y >= 0 && q.y < P.V);
    const size_t row_t = (size_t)q.b * (P.kmax + 1) + q.i;
    const size_t row_d = (size_t)q.b * P.kmax + q.i;
    const char* trow = P.target + row_t * P.t_ld * EBT;
    const char* drow = q.has_d ? P.draft + row_d * P.d_ld * EBD : nullptr;
    const int x0 = rank * P.slice;
    const int x1 = min(P.V, x0 + P.slice);
    const int xt = x0 + tid * kGroup;  // first element of this thread's group 0

    // ---------------------------------------------------------------- load slice
    Grp<EBT> tg[NG];
    Grp<EBD> dg[NG];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const int x = xt + gi * kThreads * kGroup;
      const int end = gi < P.ng ? x1 : 0;
      load_group<EBT, false>(tg[gi], trow, x, end);
      if (q.has_d) load_group<EBD, PROBS>(dg[gi], drow, x, end);
      else load_group<EBD, PROBS>(dg[gi], drow, x, 0);
    }

    const bool greedy = q.T == 0.0f;
    RowP rt, rd;
    rt.greedy = rd.greedy = greedy;
    rt.c = greedy ? 0.0f : kLog2e / q.T;
    rt.invT = rd.invT = greedy ? 0.0f : 1.0f / q.T;
    rd.c = PROBS ? 1.0f : rt.c;
    rt.Dstar = rd.Dstar = kNoFilter;

    // ----------------------------------------------- sweep 1: max + sum (or ties)
    float mt = -INFINITY, st = 0.0f, md = -INFINITY, sd = 0.0f, rmd = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      if (gi >= P.ng) break;
      float gmt = -INFINITY, gmd = -INFINITY;
#pragma unroll
      for (int e = 0; e < kGroup; ++e) {
        const float v = gval<EBT>(tg[gi], e);
        bad |= !(v <= FLT_MAX);
        gmt = fmaxf(gmt, v);
        if (q.has_d) {
          const float vd = gval<EBD>(dg[gi], e);
          bad |= PROBS ? !(vd >= 0.0f && vd <= FLT_MAX) : !(vd <= FLT_MAX);
          gmd = fmaxf(gmd, vd);
        }
      }
      rmd = fmaxf(rmd, gmd);
      if (greedy) {
        // st / sd count ties at the running maximum
        if (gmt > mt) mt = gmt, st = 0.0f;
        if (gmd > md) md = gmd, sd = 0.0f;
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          st += gval<EBT>(tg[gi], e) == mt ? 1.0f : 0.0f;
          if (q.has_d) sd += gval<EBD>(dg[gi], e) == md ? 1.0f : 0.0f;
        }
      } else {
        if (gmt > mt) {
          st = mt == -INFINITY ? 0.0f : st * ex2((mt - gmt) * rt.c);
          mt = gmt;
        }
        if (mt != -INFINITY) {
#pragma unroll
          for (int e = 0; e < kGroup; ++e) st += ex2((gval<EBT>(tg[gi], e) - mt) * rt.c);
        }
        if (q.has_d) {
          // draft weights live in the z domain: lg2(prob)/T, or the logit itself
          float gz = PROBS ? (gmd > 0.0f ? lg2(gmd) * rd.invT : -INFINITY) : gmd;
          if (gz > md) {
            sd = md == -INFINITY ? 0.0f : sd * ex2((md - gz) * rd.c);
            md = gz;
          }
          if (md != -INFINITY) {
#pragma unroll
            for (int e = 0; e < kGroup; ++e) {
              const float vd = gval<EBD>(dg[gi], e);
              const float z = PROBS ? lg2(vd) * rd.invT : vd;
              sd += ex2((z - md) * rd.c);
            }
          }
        }
      }
    }
    // warp + block combine
    const float cc_t = rt.c, cc_d = rd.c;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mt, o), s2 = __shfl_xor_sync(0xffffffffu, st, o);
      const float m3 = __shfl_xor_sync(0xffffffffu, md, o), s3 = __shfl_xor_sync(0xffffffffu, sd, o);
      if (greedy) {
        if (m2 > mt) mt = m2, st = s2; else if (m2 == mt) st += s2;
        if (m3 > md) md = m3, sd = s3; else if (m3 == md) sd += s3;
      } else {
        combine_ms(mt, st, m2, s2, cc_t);
        combine_ms(md, sd, m3, s3, cc_d);
      }
    }
    bad = __any_sync(0xffffffffu, bad);
#pragma unroll
    for (int o = 16; o; o >>= 1) rmd = fmaxf(rmd, __shfl_xor_sync(0xffffffffu, rmd, o));
    if (lane == 0) {
      sm.scratch_f[warp][0] = mt, sm.scratch_f[warp][1] = st;
      sm.scratch_f[warp][2] = md, sm.scratch_f[warp][3] = sd;
      sm.scratch_i[warp][0] = bad;
      sm.scratch_i[warp][1] = __float_as_int(rmd);
    }
    __syncthreads();
    if (tid == 0) {
      float a = sm.scratch_f[0][0], s = sm.scratch_f[0][1], c2 = sm.scratch_f[0][2], d2 = sm.scratch_f[0][3];
      int bd = sm.scratch_i[0][0];
      float rm = __int_as_float(sm.scratch_i[0][1]);
      for (int w = 1; w < kWarps; ++w) {
        rm = fmaxf(rm, __int_as_float(sm.scratch_i[w][1]));
        if (greedy) {
          if (sm.scratch_f[w][0] > a) a = sm.scratch_f[w][0], s = sm.scratch_f[w][1];
          else if (sm.scratch_f[w][0] == a) s += sm.scratch_f[w][1];
          if (sm.scratch_f[w][2] > c2) c2 = sm.scratch_f[w][2], d2 = sm.scratch_f[w][3];
          else if (sm.scratch_f[w][2] == c2) d2 += sm.scratch_f[w][3];
        } else {
          combine_ms(a, s, sm.scratch_f[w][0], sm.scratch_f[w][1], cc_t);
          combine_ms(c2, d2, sm.scratch_f[w][2], sm.scratch_f[w][3], cc_d);
        }
        bd |= sm.scratch_i[w][0];
      }
      sm.st_m[0] = a, sm.st_s[0] = s, sm.st_m[1] = c2, sm.st_s[1] = d2;
      sm.st_bad[0] = bd;
      sm.st_raw = rm;
    }
    cluster.sync();  // partials visible cluster-wide
    {
      float a = -INFINITY, s = 0.0f, c2 = -INFINITY, d2 = 0.0f, rm = -INFINITY;
      int bd = 0;
      for (int r = 0; r < C; ++r) {
        const Smem* o = cluster.map_shared_rank(&sm, r);
        const float ma = o->st_m[0], sa = o->st_s[0], mb = o->st_m[1], sb = o->st_s[1];
        if (greedy) {
          if (ma > a) a = ma, s = sa; else if (ma == a) s += sa;
          if (mb > c2) c2 = mb, d2 = sb; else if (mb == c2) d2 += sb;
        } else {
          combine_ms(a, s, ma, sa, cc_t);
          combine_ms(c2, d2, mb, sb, cc_d);
        }
        bd |= o->st_bad[0];
        rm = fmaxf(rm, o->st_raw);
      }
      rt.m = a, rt.mz = a, rt.S = s;
      rd.S = d2;
      rd.m = rm;    // raw maximum (logit or probability): defines the top-p keys
      rd.mz = c2;   // maximum in the weight domain (== rm except for probabilities, T > 0)
      bad = bd != 0;
    }
    rt.kmax = vkey<EBT>(rt.m);
    rd.kmax = vkey<EBD>(rd.m);
    rt.Z = rt.S, rd.Z = rd.S;
    rt.invZ = 1.0f / rt.Z, rd.invZ = 1.0f / rd.Z;

    bool row_bad = bad || !q.params_ok || !y_ok || rt.m == -INFINITY ||
                   (q.has_d && (PROBS ? !(rd.m > 0.0f) : rd.m == -INFINITY));

    // ---------------------------------------------------------------- top-p
    if (!row_bad && !greedy && q.top_p < 1.0f) {
      top_p_rows<EBT, EBD, PROBS, NG>(cluster, sm, tg, dg, P.ng, q.has_d, q.top_p, rt, rd);
    }

    // ---------------------------------------------------------- accept test
    // Every CTA evaluates the test identically from the same global values.
    int state;
    bool qzero = false;
    float p_y = 0.0f, q_y = 0.0f, u = 0.0f;
    if (row_bad) {
      state = SV_ROW_INVALID;
    } else if (q.has_d) {
      const float vt = EBT == 2 ? __uint_as_float((uint32_t)((const uint16_t*)trow)[q.y] << 16)
                                : ((const float*)trow)[q.y];
      const float vd = EBD == 2 ? __uint_as_float((uint32_t)((const uint16_t*)drow)[q.y] << 16)
                                : ((const float*)drow)[q.y];
      p_y = prob<EBT, false>(vt, rt);
      q_y = prob<EBD, PROBS>(vd, rd);
      const uint4 r = philox4x32_10(make_uint4(0u, (uint32_t)q.pos, q.rid, 1u), k0, k1);
      u = uniform_from_bits(r.x);
      qzero = q_y == 0.0f;
      state = (u * q_y < p_y) ? SV_ROW_ACCEPTED : SV_ROW_REJECTED;
    } else {
      state = SV_ROW_BONUS;
    }
    uint32_t* my_state = P.row_state + row_t;
    if (rank == 0 && tid == 0) {
      st_release(my_state, tag | (qzero ? kQZeroBit : 0u) | (uint32_t)state);
      if (P.debug) {
        sv_row_debug d;
        d.p_y = p_y, d.q_y = q_y, d.u = u;
        d.p_kept = greedy || rt.Dstar == kNoFilter ? 1.0f : rt.Z / rt.S;
        d.q_kept = !q.has_d || greedy || rd.Dstar == kNoFilter ? 1.0f : rd.Z / rd.S;
        d.state = state;
        d.p_thr_key = rt.Dstar == kNoFilter ? -1 : (int32_t)(rt.kmax - rt.Dstar);
        d.q_thr_key = (!q.has_d || rd.Dstar == kNoFilter) ? -1 : (int32_t)(rd.kmax - rd.Dstar);
        P.debug[row_t] = d;
      }
    }

    // -------------------------------------------------- debug: normalised rows
    if (P.probs_p && !row_bad) {
      float* out = P.probs_p + row_t * (size_t)P.V;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int x = xt + gi * kThreads * kGroup + e;
          if (gi < P.ng && x < x1) out[x] = prob<EBT, false>(gval<EBT>(tg[gi], e), rt);
        }
    }
    if (P.probs_q && q.has_d && !row_bad) {
      float* out = P.probs_q + row_d * (size_t)P.V;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int x = xt + gi * kThreads * kGroup + e;
          if (gi < P.ng && x < x1) out[x] = prob<EBD, PROBS>(gval<EBD>(dg[gi], e), rd);
        }
    }

    // --------------------------------------------- resolve: is this row the one?
    if (state != SV_ROW_ACCEPTED) {
      if (rank == 0 && tid == 0) {
        int resolver = 1;
        uint32_t st_bits = qzero ? SV_ST_Q_ZERO : 0u;
        const uint32_t* rs = P.row_state + (size_t)q.b * (P.kmax + 1);
        for (int j = 0; j < q.i && resolver == 1; ++j) {
          uint32_t w = 0;
          int spins = 0;
          for (;;) {
            w = ld_acquire(rs + j);
            if ((w & ~0xFu) == tag && (w & kStateMask) != 0) break;
            if (++spins > P.spin_limit) { resolver = 2; break; }
            __nanosleep(spins < 16 ? 32 : 256);
          }
          if (resolver == 2) break;
          if ((w & kStateMask) != SV_ROW_ACCEPTED) resolver = 0;
          if (w & kQZeroBit) st_bits |= SV_ST_Q_ZERO;
        }
        if (resolver == 2) {
          report(P.err, SV_ERR_TIMEOUT);
          write_bad_outputs(P, q.b, SV_ST_TIMEOUT);
          resolver = 0;
        }
        if (resolver == 1 && state == SV_ROW_INVALID) {
          write_bad_outputs(P, q.b, SV_ST_BAD_INPUT);
          resolver = 0;
        }
        sm.decide[0] = resolver;
        sm.decide[1] = (int)st_bits;
      }
      cluster.sync();
      const int* dc = cluster.map_shared_rank(&sm.decide[0], 0);
      const int resolver = dc[0];
      const uint32_t st_bits = (uint32_t)dc[1];
      if (resolver) {
        const bool residual = state == SV_ROW_REJECTED;
        float bw = 0.0f, bE = 1.0f;
        int bidx = 0x7FFFFFFF;
        race_slice<EBT, EBD, PROBS, NG>(tg, dg, P.ng, xt, residual, rt, rd, (uint32_t)q.pos,
                                        q.rid, k0, k1, bw, bE, bidx);
        warp_race(bw, bE, bidx);
        if (lane == 0) sm.scratch_r[warp] = {bw, bE, bidx};
        __syncthreads();
        if (tid == 0) {
          RacePart a = sm.scratch_r[0];
          for (int w = 1; w < kWarps; ++w) {
            const RacePart o = sm.scratch_r[w];
            if (better(o.w, o.E, o.idx, a.w, a.E, a.idx)) a = o;
          }
          sm.race[0] = a;
        }
        cluster.sync();
        RacePart win = cluster.map_shared_rank(&sm, 0)->race[0];
        for (int r = 1; r < C; ++r) {
          const RacePart o = cluster.map_shared_rank(&sm, r)->race[0];
          if (better(o.w, o.E, o.idx, win.w, win.E, win.idx)) win = o;
        }
        uint32_t extra = 0u;
        if (!(win.w > 0.0f)) {
          // residual numerically empty: draw from p with the same exponentials
          extra = SV_ST_RESIDUAL_EMPTY;
          bw = 0.0f, bE = 1.0f, bidx = 0x7FFFFFFF;
          race_slice<EBT, EBD, PROBS, NG>(tg, dg, P.ng, xt, false, rt, rd, (uint32_t)q.pos, q.rid,
                                          k0, k1, bw, bE, bidx);
          warp_race(bw, bE, bidx);
          if (lane == 0) sm.scratch_r[warp] = {bw, bE, bidx};
          __syncthreads();
          if (tid == 0) {
            RacePart a = sm.scratch_r[0];
            for (int w = 1; w < kWarps; ++w) {
              const RacePart o = sm.scratch_r[w];
              if (better(o.w, o.E, o.idx, a.w, a.E, a.idx)) a = o;
            }
            sm.race[1] = a;
          }
          cluster.sync();
          win = cluster.map_shared_rank(&sm, 0)->race[1];
          for (int r = 1; r < C; ++r) {
            const RacePart o = cluster.map_shared_rank(&sm, r)->race[1];
            if (better(o.w, o.E, o.idx, win.w, win.E, win.idx)) win = o;
          }
        }
        if (rank == 0 && tid == 0) {
          const int a = q.i;
          int32_t* ot = P.out_tokens + (size_t)q.b * (P.kmax + 1);
          for (int j = 0; j < a; ++j) ot[j] = P.tokens[(size_t)q.b * P.kmax + j];
          ot[a] = win.idx;
          for (int j = a + 1; j <= P.kmax; ++j) ot[j] = -1;
          P.accepted[q.b] = a;
          P.num_emitted[q.b] = a + 1;
          P.status[q.b] = st_bits | extra;
        }
      }
    }

    // next ticket, then the end-of-row barrier publishes it
    grab(parity ^ 1);
    cluster.sync();
  }

  // all peers must be done reading rank 0's shared memory before it exits
  cluster.sync();
  if (rank == 0 && tid == 0) {
    __threadfence();
    const uint32_t nclusters = gridDim.x / (uint32_t)C;
    const uint32_t d = atomicAdd(P.hdr + kHdrDone, 1u);
    if (d == nclusters - 1) {
      P.hdr[kHdrTicket] = 0u;
      P.hdr[kHdrDone] = 0u;
      __threadfence();
      atomicAdd(P.hdr + kHdrEpoch, 1u);
    }
  }
}

using KernelFn = void (*)(KParams);

// One getter per translation unit that instantiates kernel variants.
KernelFn kernel_bf16_bf16_logits();
KernelFn kernel_bf16_f32_probs();
KernelFn kernel_bf16_f32_logits();
KernelFn kernel_f32_f32_logits();
KernelFn kernel_f32_f32_probs();
KernelFn kernel_f32_bf16_logits();

size_t workspace_bytes_for(int B, int kmax);

}  // namespace sv
