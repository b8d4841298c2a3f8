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
//    the target row and, for i < k_b, the draft row.  Each CTA pulls its 1/C
//    vocabulary slice of both rows from HBM once, with 1-D TMA bulk copies
//    (cp.async.bulk, one mbarrier per 2048-element block) into shared memory,
//    and every pass (statistics, top-p histogram, race) then reads shared
//    memory in compact rolled loops; the statistics sweep starts on each block
//    as soon as it lands.  Row statistics are combined across the cluster
//    through distributed shared memory (DSMEM), one warp gathering the C
//    partials in parallel.
//  * One sweep for the statistics: per 8-element group a packed bf16x2 max,
//    then an online sum of 2^((v - m) c) with paired fp32 (f32x2) add/multiply;
//    NaN / +inf inputs surface in the sums, so no per-element check is paid.
//    Greedy rows (T = 0) count tied maxima instead.
//  * Top-p: for bf16 rows an exact 256-bin count histogram of the bf16 order
//    key below the row maximum, filled through a packed window compare; rows
//    whose boundary lies deeper (and fp32 rows) descend radix-wise.
//  * Rows are handed out by a ticket counter in (position, request) order, so
//    a row only ever waits on rows with earlier tickets, which running
//    clusters already hold (no deadlock); every wait is bounded.  A row whose
//    request already has a known earlier rejection is skipped without being
//    loaded, so the bytes read approach the rows the method needs.  Exactly
//    one row per request -- the first rejection, or the bonus row -- runs the
//    race and writes the request's outputs.
//  * The race filters whole 8-element groups by one value threshold (the
//    top-p boundary, or the bound w / E_min below the running best) before
//    any Philox work, and evaluates an accurate logf only for candidates the
//    fast MUFU estimate cannot rule out.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = 8;  // elements per group (one 16-byte bf16 vector)
constexpr int kBlk = kThreads * kGroup;  // elements per TMA block (one group per thread)
constexpr int kMaxBlk = 8;               // blocks per slice: slices hold <= 16384 elements
constexpr int64_t kMaxRepLd = 1 << 24;  // longest repetition-penalty history per request
constexpr uint32_t kNoFilter = 0xFFFFFFFFu;
constexpr int kMaxCluster = 16;
constexpr int kMaxK = 64;
constexpr int kDefaultSpin = 1 << 20;
constexpr int kWindowGuess = 2048;  // elements assumed below a top-p boundary (see top_p_rows)
constexpr float kEminSafe = 5.9604e-8f;  // <= -ln(1 - 2^-24), the smallest E

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
  int slice;      // elements per CTA (multiple of 8, <= kMaxBlk * kBlk)
  int d_off;      // byte offset of the draft slice in dynamic shared memory
  int n_tickets;  // (kmax + 1) * B
  int spin_limit;
  const int32_t* eos;      // [B] or null
  const int32_t* max_new;  // [B] or null
  const int32_t* top_k;       // [B] or null
  const float* rep_penalty;   // [B] or null
  const int32_t* rep_tokens;  // [B][rep_ld]
  int rep_ld;
  int rep_draft;  // 1: draft rows are logits and take the penalty too
};

// ---------------------------------------------------------------------------
// packed arithmetic (sm_100+: f32x2; sm_90+: bf16x2)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// bit 0: low half >= thr, bit 1: high half >= thr (NaN compares false)
__device__ __forceinline__ uint32_t bge2(uint32_t a, uint32_t thr2) {
  uint32_t r;
  asm("{.reg .pred p, q; setp.ge.bf16x2 p|q, %1, %2; selp.u32 %0, 1, 0, p; @q or.b32 %0, %0, 2;}"
      : "=r"(r)
      : "r"(a), "r"(thr2));
  return r;
}

// ---------------------------------------------------------------------------
// Groups of 8 elements in registers: 4 words of bf16 pairs or 8 fp32 words.
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

// elements (2p, 2p+1) of a group as a float pair
template <int EB>
__device__ __forceinline__ float2 gpair(const Grp<EB>& g, int p) {
  if constexpr (EB == 2) {
    const uint32_t x = g.w[p];
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
  } else {
    return make_float2(__uint_as_float(g.w[2 * p]), __uint_as_float(g.w[2 * p + 1]));
  }
}

template <int EB>
__device__ __forceinline__ float group_max(const Grp<EB>& g) {
  if constexpr (EB == 2) {
    const uint32_t m = bmax2(bmax2(g.w[0], g.w[1]), bmax2(g.w[2], g.w[3]));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  } else {
    float m = __uint_as_float(g.w[0]);
#pragma unroll
    for (int e = 1; e < 8; ++e) m = fmaxf(m, __uint_as_float(g.w[e]));
    return m;
  }
}

// 8-bit mask of the group's elements >= thr (thr2 = thr as a packed bf16 pair)
template <int EB>
__device__ __forceinline__ uint32_t group_ge(const Grp<EB>& g, float thr, uint32_t thr2) {
  uint32_t m = 0;
  if constexpr (EB == 2) {
#pragma unroll
    for (int p = 0; p < 4; ++p) m |= bge2(g.w[p], thr2) << (2 * p);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) m |= (__uint_as_float(g.w[e]) >= thr ? 1u : 0u) << e;
  }
  return m;
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

// Packed bf16 pair of the largest bf16 value <= v (v itself when v is a bf16
// value), so that "x >= pair" over bf16 x never drops an x >= v.
__device__ __forceinline__ uint32_t bf16_pair_of(float v) {
  const uint32_t u = __float_as_uint(v);
  uint32_t h = u >> 16;
  if ((u & 0x8000FFFFu) > 0x80000000u) h += 1u;  // negative with dropped bits: round down
  return h | (h << 16);
}

template <int EB, bool PROBS>
__device__ __forceinline__ uint32_t neutral_word() {
  return PROBS ? 0u : (EB == 2 ? 0xFF80FF80u : 0xFF800000u);
}

// Neutralise lanes at or beyond `end` (only the group holding the row's end).
template <int EB, bool PROBS>
__device__ __forceinline__ void mask_group(Grp<EB>& g, int x, int end) {
  if (x < end && x + kGroup > end) {
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      if (x + e >= end) {
        if constexpr (EB == 2) {
          const uint32_t n16 = PROBS ? 0u : 0xFF80u;
          uint32_t& w = g.w[e >> 1];
          w = (e & 1) ? ((w & 0x0000FFFFu) | (n16 << 16)) : ((w & 0xFFFF0000u) | n16);
        } else {
          g.w[e] = neutral_word<EB, PROBS>();
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Per-row transform parameters (identical in every CTA of the cluster).
// ---------------------------------------------------------------------------
struct RowP {
  float m;         // maximum raw value (logit, or probability)
  float mz;        // maximum in the weight domain (logit, or lg2(prob)/T)
  float c;         // weight scale: log2(e)/T for logits, 1 for probabilities
  float invT;      // 1/T (probabilities)
  bool greedy;     // T == 0
  float S;         // sum of weights over the row (T > 0) / tie count (T == 0)
  float Z;         // normaliser of the kept set
  float invZ;
  uint32_t kmax;   // vkey(m)
  uint32_t Dstar;  // kept iff vkey(m) - vkey(v) <= Dstar; kNoFilter = all
  float vstar;     // smallest kept raw value (-inf / 0 when nothing is filtered)
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

// State of one row's top-p search.
struct TopLv {
  uint32_t lo;  // distance offset of the current level's bin 0
  int shift;    // bin width 2^shift (0: exact keys)
  float above;  // mass of bins above the current range
  float R;      // target: mass top_p * S, or a count (top-k)
  int window;   // the current level is the exact bf16 count window
  int done;
  int guess;    // the window floor is the guessed one (a miss retries with the bound)
  int radix;    // the boundary came from the radix descent (kept mass recomputed)
};

struct RowRes {
  uint32_t Dstar;
  float Z, invZ, vstar;
};


// Parameters of one ticket's row, prepared by rank 0's warp 0 and read by
// every CTA of the cluster through DSMEM.
struct Ticket {
  int t, kind, kb, y, pos;
  uint32_t rid;
  float T, top_p, vt, vd;  // vt / vd: target / draft value at the proposed token
  int eos;                 // the request's end-of-sequence id, or -1
  int cap_row;             // 1: accepting this row reaches the output cap
  float theta;             // repetition penalty (1: none)
  int top_k;               // <= 0: none
};

// One warp's statistics partial: a = (target max, target sum, draft raw
// maximum, TMA failure flag), d = (draft max in the weight domain, draft sum).
struct alignas(16) StatPart {
  float4 a, d;
};

struct Smem {
  unsigned long long bar[2];  // TMA completion: target / draft slice
  Ticket tk[2];              // [iteration parity] the row to work on (rank 0 only)
  int decide[4];             // resolver decision (rank 0 only)
  StatPart part[kWarps];     // per-warp maxima partials
  StatPart cpart;            // the CTA's maxima partial, read over DSMEM
  float2 spart[kWarps];      // per-warp weight-sum partials (target, draft)
  float2 cspart;             // the CTA's weight sums, read over DSMEM
  alignas(16) uint32_t hist[2][2][256];  // [buffer][row][bin]; read as uint4 over DSMEM
  RacePart rpart[2][kWarps]; // per-warp race partials [slot]
  RacePart crpart[2];        // the CTA's race winner [slot], read over DSMEM
  union {
    uint16_t idx[kWarps][256];  // race candidates (slice element index)
    uint8_t bin[kWarps][512];   // window bins
  } wb;                         // per-warp compaction buffers
  float kz[2], kz_all[2];    // kept-mass partials (read over DSMEM) and totals
  TopLv lv[2];               // top-p search state (local broadcast)
  RowRes rres[2];            // top-p results (local broadcast)
  float scratch_f[kWarps][4];
};
static_assert(offsetof(Smem, hist) % 16 == 0, "16-byte DSMEM loads of the histograms");
static_assert(offsetof(Smem, part) % 16 == 0, "16-byte DSMEM loads of the stats partials");
static_assert(sizeof(Smem::wb) * 8 >= kMaxBlk * kBlk, "the penalty bitmap covers a slice");

enum : int { kDone = 0, kWork = 2 };

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

__device__ __forceinline__ void combine_ties(float& m, float& s, float m2, float s2) {
  if (m2 > m) m = m2, s = s2;
  else if (m2 == m) s += s2;
}

__device__ __forceinline__ uint32_t epoch_tag(uint32_t epoch) { return (epoch & 0x0FFFFFFFu) << 4; }

// Has an earlier row of request b already been decided as not accepted?
// The warp's lanes read rows j = lane, lane + 32 in parallel (i <= 64).
__device__ __forceinline__ bool warp_earlier_rejected(const KParams& P, int b, int i, uint32_t tag) {
  const uint32_t* rs = P.row_state + (size_t)b * (P.kmax + 1);
  const int lane = threadIdx.x & 31;
  bool hit = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    if (j < i) {
      const uint32_t w = ld_relaxed(rs + j);
      hit |= (w & ~0xFu) == tag && (w & kStateMask) != 0 && (w & kStateMask) != SV_ROW_ACCEPTED;
    }
  }
  return __any_sync(0xffffffffu, hit);
}

static __device__ void write_bad_outputs(const KParams& P, int b, uint32_t st) {
  P.accepted[b] = -1;
  P.num_emitted[b] = 0;
  P.status[b] = st;
  for (int j = 0; j <= P.kmax; ++j) P.out_tokens[(size_t)b * (P.kmax + 1) + j] = -1;
}

// ---------------------------------------------------------------------------
// TMA bulk copies and mbarriers (1-D, no tensor map, no multicast)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Pull [src, src + bytes) into L2 without waiting (bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// try_wait with a suspend-time hint: the warp is parked until the phase
// completes (or ~0.5 ms pass) instead of spinning through issue slots.
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 500000; selp.u32 %0, 1, 0, p;}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok;
}

// Bounded wait for a TMA block (at most ~1 s); returns false (and reports) if
// it never lands.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity, int* err) {
  for (int it = 0; it < 2000; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  report(err, SV_ERR_TIMEOUT);
  return false;
}

// One 8-element group of this thread from the shared-memory slice starting at
// element x0 (lanes at or beyond x1 neutralised).
template <int EB, bool PROBS>
__device__ __forceinline__ void lds_group(Grp<EB>& g, const char* sbase, int x0, int x, int x1) {
  const uint4* p = reinterpret_cast<const uint4*>(sbase + (size_t)(x - x0) * EB);
  const uint4 a = p[0];
  g.w[0] = a.x, g.w[1] = a.y, g.w[2] = a.z, g.w[3] = a.w;
  if constexpr (EB == 4) {
    const uint4 b = p[1];
    g.w[4] = b.x, g.w[5] = b.y, g.w[6] = b.z, g.w[7] = b.w;
  }
  mask_group<EB, PROBS>(g, x, x1);
}

template <int EB, bool PROBS>
__device__ __forceinline__ void lds_group_or_neutral(Grp<EB>& g, const char* sbase, int x0, int x,
                                                     int x1) {
  if (x < x1) {
    lds_group<EB, PROBS>(g, sbase, x0, x, x1);
  } else {
#pragma unroll
    for (int j = 0; j < EB * 2; ++j) g.w[j] = neutral_word<EB, PROBS>();
  }
}

// The thread's groups of a slice: group k starts at element x0 + k*kBlk + tid*8.
// stride: elements between a thread's consecutive groups (threads x 8);
// tid: the thread's index among the threads that share the slice.
struct SliceIter {
  int x0, x1, nblk, V;
  int stride, tid;
  __device__ __forceinline__ int x(int blk) const { return x0 + blk * stride + tid * kGroup; }
};

// ---------------------------------------------------------------------------
// per-group passes
// ---------------------------------------------------------------------------
// Row statistics in two sweeps over the thread's groups: the raw maximum as
// the TMA blocks land, then the weight sum relative to the thread's own
// maximum.  Logit rows: weight 2^((v - mz) c) with mz = max v.  Probability
// rows: z = lg2(v)/T, weight 2^(z - mz).  T = 0: the count of elements equal
// to the maximum.  Partials meet in warp_ms / cluster_ms, which rescale
// each sum to the common maximum.
template <int EB>
__device__ __forceinline__ void max_group(const Grp<EB>& g, uint32_t& mx2, float& mx) {
  if constexpr (EB == 2) {
    mx2 = bmax2(mx2, bmax2(bmax2(g.w[0], g.w[1]), bmax2(g.w[2], g.w[3])));
  } else {
    const float a = fmaxf(fmaxf(__uint_as_float(g.w[0]), __uint_as_float(g.w[1])),
                          fmaxf(__uint_as_float(g.w[2]), __uint_as_float(g.w[3])));
    const float b = fmaxf(fmaxf(__uint_as_float(g.w[4]), __uint_as_float(g.w[5])),
                          fmaxf(__uint_as_float(g.w[6]), __uint_as_float(g.w[7])));
    mx = fmaxf(mx, fmaxf(a, b));
  }
}

template <int EB>
__device__ __forceinline__ float max_value(uint32_t mx2, float mx) {
  if constexpr (EB == 2) return fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u));
  else return mx;
}

// Sum of one group's weights.  A value no weight formula reads (NaN; for
// probability rows also a negative value) turns the sum into NaN, which the
// row's validity check catches.
template <int EB, bool PROBS>
__device__ __forceinline__ float sum_group(const Grp<EB>& g, bool greedy, float mz, float c,
                                           float invT) {
  const float kNaN = __int_as_float(0x7FC00000);
  if (greedy) {
    float n = 0.0f;
    bool bad = false;
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      const float v = gval<EB>(g, e);
      n += v == mz ? 1.0f : 0.0f;
      bad |= !(v >= (PROBS ? 0.0f : -INFINITY));
    }
    return bad ? kNaN : n;
  }
  if (mz == -INFINITY) {  // the thread holds no weight: only neutral values are valid
    bool bad = false;
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      const float v = gval<EB>(g, e);
      bad |= PROBS ? !(v == 0.0f) : !(v == -INFINITY);
    }
    return bad ? kNaN : 0.0f;
  }
  float2 a = make_float2(0.0f, 0.0f), b = a;
  if constexpr (!PROBS) {
    const float2 nm = make_float2(-mz, -mz), cc = make_float2(c, c);
    const float2 d0 = f2mul(f2add(gpair<EB>(g, 0), nm), cc);
    const float2 d1 = f2mul(f2add(gpair<EB>(g, 1), nm), cc);
    const float2 d2 = f2mul(f2add(gpair<EB>(g, 2), nm), cc);
    const float2 d3 = f2mul(f2add(gpair<EB>(g, 3), nm), cc);
    a = f2add(make_float2(ex2(d0.x), ex2(d0.y)), make_float2(ex2(d1.x), ex2(d1.y)));
    b = f2add(make_float2(ex2(d2.x), ex2(d2.y)), make_float2(ex2(d3.x), ex2(d3.y)));
  } else {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 v = gpair<EB>(g, p);
      const float2 e = make_float2(ex2(lg2(v.x) * invT - mz), ex2(lg2(v.y) * invT - mz));
      if (p < 2) a = f2add(a, e);
      else b = f2add(b, e);
    }
  }
  const float2 t = f2add(a, b);
  return t.x + t.y;
}

// Scale a (max, sum) partial to the common maximum M.  A partial without
// elements (sum 0) stays 0 whatever its maximum.
__device__ __forceinline__ float rescale(float m, float s, float M, float c, bool greedy) {
  if (greedy) return (m == M || s != s) ? s : 0.0f;  // a NaN partial must survive
  return s == 0.0f ? 0.0f : s * ex2((m - M) * c);
}

// All lanes end with the same (M, S): butterfly max, then butterfly sum.
__device__ __forceinline__ void warp_ms(float& m, float& s, float c, bool greedy) {
  float M = m;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = rescale(m, s, M, c, greedy);
#pragma unroll
  for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  m = M, s = S;
}

// Combine stats partials held one per lane (lanes without one hold the
// neutral partial): a = (target max, target sum, draft raw maximum, failure
// flag), d = (draft max, draft sum).  Every lane ends with the same result.
template <bool PROBS>
__device__ __forceinline__ StatPart neutral_part() {
  return {make_float4(-INFINITY, 0.0f, PROBS ? 0.0f : -INFINITY, 0.0f),
          make_float4(-INFINITY, 0.0f, 0.0f, 0.0f)};
}

__device__ __forceinline__ StatPart combine_parts(const StatPart& v, float ct, float cd, bool greedy) {
  float Mt = v.a.x, Md = v.d.x, Rm = v.a.z, bad = v.a.w;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, o));
    Md = fmaxf(Md, __shfl_xor_sync(0xffffffffu, Md, o));
    Rm = fmaxf(Rm, __shfl_xor_sync(0xffffffffu, Rm, o));
    bad = fmaxf(bad, __shfl_xor_sync(0xffffffffu, bad, o));
  }
  float St = rescale(v.a.x, v.a.y, Mt, ct, greedy), Sd = rescale(v.d.x, v.d.y, Md, cd, greedy);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    St += __shfl_xor_sync(0xffffffffu, St, o);
    Sd += __shfl_xor_sync(0xffffffffu, Sd, o);
  }
  return {make_float4(Mt, St, Rm, bad), make_float4(Md, Sd, 0.0f, 0.0f)};
}

// Warp-inclusive scan of a per-lane count.
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__device__ __forceinline__ void flush_bins(uint32_t* hist, const uint8_t* wb, int total) {
  __syncwarp();
  for (int j = threadIdx.x & 31; j < total; j += 32) {
    atomicAdd(&hist[wb[j]], 1u);  // a byte: always inside the 256 bins
  }
  __syncwarp();
}

// One 16-byte group of a bf16 slice; a group starting at or past the slice end
// reads the slice's first group instead (callers mask it out).
__device__ __forceinline__ uint4 load_group_bf16(const char* s, const SliceIter& it, int blk) {
  const int x = it.x(blk);
  return *reinterpret_cast<const uint4*>(s + (size_t)(x < it.x1 ? x - it.x0 : 0) * 2);
}

__device__ __forceinline__ uint32_t bf16_order_key(uint32_t b16) {
  if (b16 == 0x8000u) b16 = 0u;  // -0 keys like +0
  return b16 ^ ((b16 & 0x8000u) ? 0xFFFFu : 0x8000u);
}

// Exact window histogram for bf16 rows: count elements by bf16 order-key
// distance D = kmax - key(v) for keys in [lo_key, kmax] (one bin per bf16
// value, at most 256).  The thread's 8 groups are loaded together and turned
// into 64 candidate bits; one warp scan places the candidates in the warp's
// buffer and the atomics run on full warps.  The candidate walk is a single
// loop that re-reads each hit from shared memory: unrolled copies of it made
// the code large enough that instruction fetch dominated.  A window too dense
// for the buffer goes one group column at a time.
// Candidate bits of one bf16 group: element e >= the floor pair thr2 (bit e),
// lanes at or past the row end dropped.
__device__ __forceinline__ uint32_t window_bits_bf16(const uint4& g, uint32_t thr2, int x, int x1) {
  uint32_t m = bge2(g.x, thr2) | (bge2(g.y, thr2) << 2) | (bge2(g.z, thr2) << 4) |
               (bge2(g.w, thr2) << 6);
  if (x + kGroup > x1) m = x < x1 ? m & ((1u << (x1 - x)) - 1u) : 0u;  // past the end
  return m;
}

// Histogram the candidates of the thread's 8 groups (bits mlo: groups 0-3,
// mhi: groups 4-7; cnt of them).  One warp scan places the candidates in the
// warp's buffer and the atomics run on full warps.  The candidate walk is a
// single loop that re-reads each hit from shared memory: unrolled copies of
// it made the code large enough that instruction fetch dominated.  A window
// too dense for the buffer goes one group column at a time.
__device__ __forceinline__ void window_commit_bf16(const char* s, uint32_t kmax, uint32_t mlo,
                                                   uint32_t mhi, int cnt, const SliceIter& it,
                                                   uint32_t* hist, uint8_t* wb) {
  const int incl = warp_incl_scan(cnt);
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total == 0) return;
  const uint16_t* sv = reinterpret_cast<const uint16_t*>(s);
  const int base = it.tid * kGroup;  // slice offset of this thread's group 0
  unsigned long long mk = ((unsigned long long)mhi << 32) | mlo;
  if (total <= 512) {
    int pos = incl - cnt;
    while (mk) {
      const int bit = __ffsll((long long)mk) - 1;
      mk &= mk - 1ull;
      const uint32_t key = bf16_order_key(sv[base + (bit >> 3) * it.stride + (bit & 7)]);
      wb[pos++] = (uint8_t)(kmax - key);
    }
    flush_bins(hist, wb, total);
    return;
  }
#pragma unroll 1
  for (int blk = 0; blk < it.nblk; ++blk) {  // dense window: one group column at a time
    uint32_t m = (uint32_t)(mk >> (8 * blk)) & 0xFFu;
    const int n = __popc(m);
    const int inc = warp_incl_scan(n);
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    if (tot == 0) continue;
    int pos = inc - n;
    while (m) {
      const int e = __ffs(m) - 1;
      m &= m - 1;
      const uint32_t key = bf16_order_key(sv[base + blk * it.stride + e]);
      wb[pos++] = (uint8_t)(kmax - key);
    }
    flush_bins(hist, wb, tot);
  }
}

// Exact window histogram for bf16 rows: count elements by bf16 order-key
// distance D = kmax - key(v) for keys in [lo_key, kmax] (one bin per bf16
// value, at most 256).  The thread's 8 groups are loaded together (their
// latencies overlap) and turned into candidate bits.
__device__ __forceinline__ void window_row_bf16(const char* s, const SliceIter& it, uint32_t kmax,
                                                uint32_t lo_key, uint32_t* hist, uint8_t* wb) {
  const uint32_t thr2 = bf16_pair_of(vkey_value<2>(lo_key));
  uint4 g[kMaxBlk];
#pragma unroll
  for (int blk = 0; blk < kMaxBlk; ++blk) g[blk] = load_group_bf16(s, it, blk);
  uint32_t mlo = 0u, mhi = 0u;
  int cnt = 0;
#pragma unroll
  for (int blk = 0; blk < kMaxBlk; ++blk) {
    const uint32_t m = window_bits_bf16(g[blk], thr2, it.x(blk), it.x1);
    cnt += __popc(m);
    if (blk < 4) mlo |= m << (8 * blk);
    else mhi |= m << (8 * (blk - 4));
  }
  window_commit_bf16(s, kmax, mlo, mhi, cnt, it, hist, wb);
}

// Lowest key a top-p boundary can have when at most n elements lie below it:
// every element below value v_lo weighs at most w(v_lo) = (1 - top_p) S / (2 n),
// so together they hold at most half the excluded mass and the boundary lies
// at or above v_lo.  With n = V this is a bound; clamped to the 256-bin window
// below kmax.
__device__ __forceinline__ uint32_t window_lo_key_x(const RowP& r, float excl, int n) {
  const uint32_t floor_key = r.kmax >= 255u ? r.kmax - 255u : 0u;
  const float wlo = excl / (2.0f * (float)n);
  if (!(wlo > 0.0f)) return floor_key;
  const float vlo = r.m + lg2(wlo) / r.c - 1.0f / r.c;  // one log2 unit of slack
  if (!(vlo > -FLT_MAX)) return floor_key;
  // bf16 value at or below vlo, as a key
  const uint32_t pair = bf16_pair_of(vlo);
  const uint32_t k = vkey<2>(__uint_as_float(pair << 16));
  return k > floor_key ? k : floor_key;
}

// The same with the excluded mass (1 - top_p) S of a plain top-p row.
__device__ __forceinline__ uint32_t window_lo_key(const RowP& r, float top_p, int n) {
  return window_lo_key_x(r, (1.0f - top_p) * r.S, n);
}

// General histogram level: every element whose distance D lies in
// [lo, lo + 256 << shift) adds its weight (top-k: 1) to bin (D - lo) >> shift.
template <int EB, bool PROBS, bool CNT>
__device__ __forceinline__ void level_group(const Grp<EB>& g, const RowP& r, uint32_t lo, int shift,
                                            uint32_t* hist) {
  const uint32_t span = shift >= 24 ? 0xFFFFFFFFu : ((256u << shift) - 1u);
#pragma unroll
  for (int e = 0; e < kGroup; ++e) {
    const float v = gval<EB>(g, e);
    const uint32_t D = r.kmax - vkey<EB>(v);
    const uint32_t u = D - lo;
    if (D >= lo && u <= span && v > (PROBS ? 0.0f : -INFINITY))
      atomicAdd(reinterpret_cast<float*>(&hist[u >> shift]), CNT ? 1.0f : weight<PROBS>(v, r));
  }
}

// One warp resolves one level of one row: gathers the C ranks' 256-bin
// histograms (lane l owns bins 8l .. 8l+7; the remote loads of four ranks
// are in flight together), scans them in the warp, and picks the boundary bin.  Every CTA
// runs the same arithmetic on the same data, so all reach the same result.
template <int EB, bool PROBS, bool CNT>
__device__ __forceinline__ void resolve_level(cg::cluster_group& cluster, const uint32_t* hist, int C,
                                              TopLv& lv, RowP& r) {
  const int lane = threadIdx.x & 31;
  float h[8];  // counts (exact in fp32 below 2^24) or weights per bin
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = 0.0f;
#pragma unroll
  for (int q0 = 0; q0 < kMaxCluster; q0 += 4) {
    if (q0 < C) {
      uint4 a[4], b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q0 + q < C) {
          const uint4* src = reinterpret_cast<const uint4*>(cluster.map_shared_rank(hist, q0 + q)) + 2 * lane;
          a[q] = src[0], b[q] = src[1];
        } else {
          a[q] = make_uint4(0u, 0u, 0u, 0u), b[q] = a[q];
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // rank order
        const uint32_t w[8] = {a[q].x, a[q].y, a[q].z, a[q].w, b[q].x, b[q].y, b[q].z, b[q].w};
#pragma unroll
        for (int k = 0; k < 8; ++k) h[k] += lv.window ? (float)w[k] : __uint_as_float(w[k]);
      }
    }
  }
  if (lv.window && !CNT) {  // counts to weights (top-k keeps the counts)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      h[k] = h[k] > 0.0f ? h[k] * weight<PROBS>(vkey_value<2>(r.kmax - (uint32_t)(8 * lane + k)), r) : 0.0f;
  }
  float inc[8], t = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) t += h[k], inc[k] = t;
  float off = t;  // warp exclusive scan of the lane totals
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_up_sync(0xffffffffu, off, o);
    if (lane >= o) off += v;
  }
  off -= t;
  int first = 8;
#pragma unroll
  for (int k = 7; k >= 0; --k)
    if (lv.above + off + inc[k] >= lv.R) first = k;
  const uint32_t hit = __ballot_sync(0xffffffffu, first < 8);
  int c;
  float cexcl, ch;
  if (hit) {
    const int src = __ffs(hit) - 1;
    float my_excl = off, my_h = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k == first) my_h = h[k], my_excl = off + inc[k] - h[k];
    c = 8 * src + __shfl_sync(0xffffffffu, first, src);
    cexcl = __shfl_sync(0xffffffffu, my_excl, src);
    ch = __shfl_sync(0xffffffffu, my_h, src);
  } else if (lv.window && lv.guess) {  // boundary below the guessed floor: retry with the bound
    lv.guess = 0;
    return;
  } else if (lv.window) {  // boundary beyond the exact window: full radix descent
    lv.window = 0;
    lv.radix = 1;
    lv.lo = 0u;
    lv.above = 0.0f;
    lv.shift = EB == 2 ? 8 : 24;
    return;
  } else {  // rounding left the target mass unreachable: keep through the last non-empty bin
    int last = -1;
    float my_excl = 0.0f, my_h = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (h[k] > 0.0f) last = k, my_h = h[k], my_excl = off + inc[k] - h[k];
    const uint32_t any = __ballot_sync(0xffffffffu, last >= 0);
    const int src = any ? 31 - __clz(any) : 0;
    c = any ? 8 * src + __shfl_sync(0xffffffffu, last, src) : 0;
    cexcl = __shfl_sync(0xffffffffu, my_excl, src);
    ch = __shfl_sync(0xffffffffu, my_h, src);
  }
  lv.above += cexcl;
  lv.lo += (uint32_t)c << lv.shift;
  if (lv.shift == 0) {
    r.Dstar = lv.lo;
    r.Z = lv.above + ch;
    r.invZ = 1.0f / r.Z;
    r.vstar = vkey_value<EB>(r.kmax - r.Dstar);
    lv.done = 1;
  } else {
    lv.shift -= 8;
  }
}

// Top-p threshold of the target row and (if has_d) the draft row held in
// shared memory across the cluster: the largest boundary whose kept mass
// reaches Rt / Rd (a window floor may assume the rows exclude at least Xt / Xd
// of their mass).  With cnt the targets are a count instead (top-k: the
// boundary keeps at least that many elements) and the kept mass is summed
// afterwards.  Sets Dstar, Z, invZ, vstar.  All control flow depends only on
// cluster-reduced values, so every CTA takes the same path.
template <int EBT, int EBD, bool PROBS, bool CNT>
__device__ __noinline__ void top_p_rows(cg::cluster_group& cluster, Smem& sm, const char* st,
                                        const char* sd, const SliceIter& it, bool has_d,
                                        float Rt, float Rd, float Xt, float Xd,
                                        RowP& rt, RowP& rd, bool pre_t, bool pre_d) {
  const int C = cluster.num_blocks();
  const int tid = threadIdx.x;
  constexpr bool cnt = CNT;
  TopLv L[2];
  L[0] = {0u, EBT == 2 ? 0 : 24, 0.0f, Rt, EBT == 2, 0, EBT == 2 && !cnt, EBT != 2};
  L[1] = {0u, EBD == 2 ? 0 : 24, 0.0f, Rd, EBD == 2 && !PROBS, !has_d,
          EBD == 2 && !PROBS && !cnt, !(EBD == 2 && !PROBS)};
  // window floors as distances below the row maxima (bf16 rows only)
  uint32_t lo_t = 255u, lo_d = 255u;
  // The first floor assumes at most kWindowGuess elements below the boundary
  // instead of V: usually true, and far fewer elements land in the window.
  // When the boundary is not inside that window, resolve_level retries with
  // the bound (n = V) and then falls back to the exact radix descent, so the
  // result never depends on the guess.
  // A row whose first window the caller already counted into sm.hist[0]
  // (pre_t / pre_d, visible cluster-wide) goes straight to its resolve.
  const int nguess = min(it.V, kWindowGuess);
  int buf = 0;
  for (bool first = true; !(L[0].done && L[1].done); first = false) {
    const bool bt = !L[0].done && !(first && pre_t);  // rows counted in this round
    const bool bd = !L[1].done && !(first && pre_d);
    if (bt || bd) {
    // (top-k: the whole 256-value window below the maximum)
    if constexpr (EBT == 2)
      lo_t = rt.kmax - (cnt ? (rt.kmax >= 255u ? rt.kmax - 255u : 0u)
                            : window_lo_key_x(rt, Xt, L[0].guess ? nguess : it.V));
    if constexpr (EBD == 2 && !PROBS)
      lo_d = rd.kmax - (cnt ? (rd.kmax >= 255u ? rd.kmax - 255u : 0u)
                            : window_lo_key_x(rd, Xd, L[1].guess ? nguess : it.V));
    if (bt) for (int j = tid; j < 256; j += kThreads) sm.hist[buf][0][j] = 0u;
    if (bd) for (int j = tid; j < 256; j += kThreads) sm.hist[buf][1][j] = 0u;
    __syncthreads();
    if constexpr (EBT == 2) {
      if (bt && L[0].window)
        window_row_bf16(st, it, rt.kmax, rt.kmax - lo_t, sm.hist[buf][0], sm.wb.bin[tid >> 5]);
    }
    if constexpr (EBD == 2 && !PROBS) {
      if (bd && L[1].window)
        window_row_bf16(sd, it, rd.kmax, rd.kmax - lo_d, sm.hist[buf][1], sm.wb.bin[tid >> 5]);
    }
    const bool gen_t = bt && !(EBT == 2 && L[0].window);
    const bool gen_d = bd && !(EBD == 2 && !PROBS && L[1].window);
    if (gen_t || gen_d) {
#pragma unroll 1
      for (int blk = 0; blk < it.nblk; ++blk) {
        const int x = it.x(blk);
        if (x >= it.x1) break;
        if (gen_t) {
          Grp<EBT> g;
          lds_group<EBT, false>(g, st, it.x0, x, it.x1);
          level_group<EBT, false, CNT>(g, rt, L[0].lo, L[0].shift, sm.hist[buf][0]);
        }
        if (gen_d) {
          Grp<EBD> g;
          lds_group<EBD, PROBS>(g, sd, it.x0, x, it.x1);
          level_group<EBD, PROBS, CNT>(g, rd, L[1].lo, L[1].shift, sm.hist[buf][1]);
        }
      }
    }
    __syncthreads();
    cluster.sync();
    }
    // warp 0 resolves the target row, warp 1 the draft row; one barrier
    // publishes both results to the whole CTA
    const int warp = tid >> 5;
    if (warp == 0 && !L[0].done) {
      resolve_level<EBT, false, CNT>(cluster, &sm.hist[buf][0][0], C, L[0], rt);
      if ((tid & 31) == 0) sm.lv[0] = L[0], sm.rres[0] = {rt.Dstar, rt.Z, rt.invZ, rt.vstar};
    }
    if (warp == 1 && !L[1].done) {
      resolve_level<EBD, PROBS, CNT>(cluster, &sm.hist[buf][1][0], C, L[1], rd);
      if ((tid & 31) == 0) sm.lv[1] = L[1], sm.rres[1] = {rd.Dstar, rd.Z, rd.invZ, rd.vstar};
    }
    __syncthreads();
    if (!L[0].done) {
      L[0] = sm.lv[0];
      rt.Dstar = sm.rres[0].Dstar, rt.Z = sm.rres[0].Z, rt.invZ = sm.rres[0].invZ, rt.vstar = sm.rres[0].vstar;
    }
    if (!L[1].done) {
      L[1] = sm.lv[1];
      rd.Dstar = sm.rres[1].Dstar, rd.Z = sm.rres[1].Z, rd.invZ = sm.rres[1].invZ, rd.vstar = sm.rres[1].vstar;
    }
    __syncthreads();  // sm.lv / sm.rres are rewritten by the next level
    buf ^= 1;
  }
  // A boundary from the radix descent comes with a kept mass summed by float
  // atomics, whose rounding grows with the number of elements sharing a bin
  // (a plateau of tied values).  Recompute it as per-thread sums reduced in a
  // fixed order across the cluster, as the row sum S is.  A top-k boundary
  // comes with a count only: its mass is summed the same way.
  const bool fix_t = L[0].radix || cnt, fix_d = has_d && (L[1].radix || cnt);
  if (fix_t || fix_d) {
    float zt = 0.0f, zd = 0.0f;
#pragma unroll 1
    for (int blk = 0; blk < it.nblk; ++blk) {
      const int x = it.x(blk);
      if (x >= it.x1) break;
      if (fix_t) {
        Grp<EBT> g;
        lds_group<EBT, false>(g, st, it.x0, x, it.x1);
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const float v = gval<EBT>(g, e);
          if (kept<EBT>(v, rt)) zt += weight<false>(v, rt);
        }
      }
      if (fix_d) {
        Grp<EBD> g;
        lds_group<EBD, PROBS>(g, sd, it.x0, x, it.x1);
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const float v = gval<EBD>(g, e);
          if (kept<EBD>(v, rd)) zd += weight<PROBS>(v, rd);
        }
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      zt += __shfl_xor_sync(0xffffffffu, zt, o);
      zd += __shfl_xor_sync(0xffffffffu, zd, o);
    }
    const int warp = tid >> 5;
    if ((tid & 31) == 0) sm.scratch_f[warp][0] = zt, sm.scratch_f[warp][1] = zd;
    __syncthreads();
    if (tid == 0) {
      float a = 0.0f, b = 0.0f;
      for (int w = 0; w < kWarps; ++w) a += sm.scratch_f[w][0], b += sm.scratch_f[w][1];
      sm.kz[0] = a, sm.kz[1] = b;
    }
    cluster.sync();
    if (tid == 0) {
      float a = 0.0f, b = 0.0f;
      for (int r = 0; r < C; ++r) {  // rank order: the same sum in every CTA
        const Smem* o = cluster.map_shared_rank(&sm, r);
        a += o->kz[0], b += o->kz[1];
      }
      sm.kz_all[0] = a, sm.kz_all[1] = b;
    }
    __syncthreads();
    if (fix_t) rt.Z = sm.kz_all[0], rt.invZ = 1.0f / rt.Z;
    if (fix_d) rd.Z = sm.kz_all[1], rd.invZ = 1.0f / rd.Z;
    cluster.sync();  // peers are done reading kz before it can be rewritten
  }
}

// The row filters: top-k (top_k > 0) and then top-p on the renormalised
// top-k rows, or top-p alone.  One call site in the row loop keeps the loop's
// register allocation independent of the filters.
template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void filter_rows(cg::cluster_group& cluster, Smem& sm, const char* st,
                                         const char* sd, const SliceIter& it, bool has_d, float top_p,
                                         int top_k, RowP& rt, RowP& rd, bool pre_t, bool pre_d) {
  if (top_k <= 0) {
    top_p_rows<EBT, EBD, PROBS, false>(cluster, sm, st, sd, it, has_d, top_p * rt.S, top_p * rd.S,
                                       (1.0f - top_p) * rt.S, (1.0f - top_p) * rd.S, rt, rd, pre_t,
                                       pre_d);
    return;
  }
  const float K = (float)top_k;
  top_p_rows<EBT, EBD, PROBS, true>(cluster, sm, st, sd, it, has_d, K, K, 0.0f, 0.0f, rt, rd, false,
                                    false);
  if (top_p < 1.0f) {
    // the boundary keeps top_p of the top-k mass, so it lies at or above the
    // top-k boundary (rounding aside: then the top-k boundary stands)
    const RowRes kt = {rt.Dstar, rt.Z, rt.invZ, rt.vstar}, kd = {rd.Dstar, rd.Z, rd.invZ, rd.vstar};
    const float Rt = top_p * kt.Z, Rd = top_p * kd.Z;
    top_p_rows<EBT, EBD, PROBS, false>(cluster, sm, st, sd, it, has_d, Rt, Rd, rt.S - Rt, rd.S - Rd,
                                       rt, rd, false, false);
    if (rt.Dstar > kt.Dstar) rt.Dstar = kt.Dstar, rt.Z = kt.Z, rt.invZ = kt.invZ, rt.vstar = kt.vstar;
    if (has_d && rd.Dstar > kd.Dstar)
      rd.Dstar = kd.Dstar, rd.Z = kd.Z, rd.invZ = kd.invZ, rd.vstar = kd.vstar;
  }
}

// Smallest target value that can still beat the running best (bw / bE): its
// weight must reach bw E_min / bE (bonus) or that times Z (residual, w <= p).
__device__ __forceinline__ float race_threshold(const RowP& rt, bool residual, float bw, float bE) {
  if (rt.greedy) return rt.m;  // only tied maxima carry weight
  const float base = rt.vstar;
  if (!(bw > 0.0f)) return base;
  float theta = bw * kEminSafe / bE;  // a smaller w cannot win
  if (residual) theta *= rt.Z;        // p = weight / Z >= w
  const float v = rt.m + lg2(theta) / rt.c - 1.0f / rt.c;  // one log2 unit of slack
  return fmaxf(base, v);
}

// Race weight of slice element j: bonus w = kept target weight (unnormalised),
// residual w = max(0, p - q).
template <int EBT, int EBD, bool PROBS>
__device__ __forceinline__ float race_weight(const char* st, const char* sd, int j, bool residual,
                                             const RowP& rt, const RowP& rd) {
  const float vp = EBT == 2 ? __uint_as_float((uint32_t)((const uint16_t*)st)[j] << 16)
                            : ((const float*)st)[j];
  if (!residual) return kept<EBT>(vp, rt) ? weight<false>(vp, rt) : 0.0f;
  const float vq = EBD == 2 ? __uint_as_float((uint32_t)((const uint16_t*)sd)[j] << 16)
                            : ((const float*)sd)[j];
  return fmaxf(0.0f, prob<EBT, false>(vp, rt) - prob<EBD, PROBS>(vq, rd));
}

// Exponential race over this warp's groups of the shared-memory slices.  The
// warp compacts candidate elements (target value >= the running threshold)
// into its buffer and processes them one per lane: one Philox draw per
// candidate, the fast E first and an accurate logf only for contenders.  The
// threshold rises with the warp's best after every flush.
template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void race_slice(const char* st, const char* sd, const SliceIter& it_ref,
                                        bool residual, const RowP& rt_ref, const RowP& rd_ref,
                                        uint32_t pos, uint32_t rid, uint32_t k0, uint32_t k1,
                                        uint16_t* wb, RacePart& best) {
  // Register copies of the caller's records: they live in its stack frame
  // (their address is passed), and the candidate loop would otherwise reload
  // them from local memory, which misses L1 beside the large slices.
  const SliceIter it = it_ref;
  const RowP rt = rt_ref, rd = rd_ref;
  const int lane = threadIdx.x & 31;
  float bw = best.w, bE = best.E;
  int bidx = best.idx;
  float vthr = race_threshold(rt, residual, bw, bE);
  int fill = 0;
  auto flush = [&]() {  // process wb[0, fill) one candidate per lane
    __syncwarp();
    for (int j = lane; j < fill; j += 32) {
      const int e = wb[j];
      const float w = race_weight<EBT, EBD, PROBS>(st, sd, e, residual, rt, rd);
      if (!(w * bE > bw * kEminSafe)) continue;
      const int x = it.x0 + e;
      const uint4 r = philox4x32_10(make_uint4((uint32_t)x >> 2, pos, rid, 0u), k0, k1);
      const uint32_t sel = (x & 3) == 0 ? r.x : (x & 3) == 1 ? r.y : (x & 3) == 2 ? r.z : r.w;
      const float U = uniform_from_bits(sel);
      const float Ef = -lg2(U) * kLn2;
      const float Elo = Ef * (1.0f - 2e-6f) - 2e-7f;  // lower bound of the exact E
      if (Elo <= 0.0f || w * bE > bw * Elo) {
        const float E = -logf(U);
        if (better(w, E, x, bw, bE, bidx)) bw = w, bE = E, bidx = x;
      }
    }
    __syncwarp();
    warp_race(bw, bE, bidx);  // the warp shares its best: a tighter threshold
    vthr = race_threshold(rt, residual, bw, bE);
    fill = 0;
  };
  // candidate masks of all of this thread's groups, then one warp scan
  uint32_t m_lo = 0, m_hi = 0;
  int cnt = 0;
#pragma unroll
  for (int blk = 0; blk < kMaxBlk; ++blk) {
    if (blk < it.nblk) {
      const int x = it.x(blk);
      uint32_t msk = 0;
      if (x < it.x1) {
        Grp<EBT> tg;
        lds_group<EBT, false>(tg, st, it.x0, x, it.x1);
        msk = group_ge<EBT>(tg, vthr, bf16_pair_of(vthr));
        // candidates are re-read from shared memory by index: drop lanes past the row end
        if (x + kGroup > it.x1) msk &= (1u << (it.x1 - x)) - 1u;
      }
      cnt += __popc(msk);
      if (blk < 4) m_lo |= msk << (8 * blk);
      else m_hi |= msk << (8 * (blk - 4));
    }
  }
  const int base = it.tid * kGroup;  // slice offset of this thread's group 0
  auto emit = [&](uint32_t m, int half, int pos) {
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      wb[pos++] = (uint16_t)(base + (half * 4 + (bit >> 3)) * it.stride + (bit & 7));
    }
  };
  const int incl = warp_incl_scan(cnt);
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total <= 256) {
    if (total) {
      const int pos = incl - cnt;
      emit(m_lo, 0, pos);
      emit(m_hi, 1, pos + __popc(m_lo));
      fill = total;
      flush();
    }
  } else {
    // dense candidates (no nucleus to filter by): every lane works through its
    // own groups with one Philox call per 4 consecutive tokens, and the warp
    // shares its best after every group column to raise the bound
#pragma unroll 1
    for (int blk = 0; blk < it.nblk; ++blk) {
      const int x = it.x(blk);
      if (x < it.x1) {
        Grp<EBT> tg;
        Grp<EBD> dg;
        lds_group<EBT, false>(tg, st, it.x0, x, it.x1);  // lanes past the end are neutral
        if (residual) lds_group<EBD, PROBS>(dg, sd, it.x0, x, it.x1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = h * 4 + j;
            const float vp = gval<EBT>(tg, e);
            w[j] = residual ? fmaxf(0.0f, prob<EBT, false>(vp, rt) - prob<EBD, PROBS>(gval<EBD>(dg, e), rd))
                            : (kept<EBT>(vp, rt) ? weight<false>(vp, rt) : 0.0f);
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
              if (better(w[j], E, x4 + j, bw, bE, bidx)) bw = w[j], bE = E, bidx = x4 + j;
            }
          }
        }
      }
      warp_race(bw, bE, bidx);
    }
  }
  best = {bw, bE, bidx};
}

// Block + cluster argmax of the race partials in slot `slot`: warp winners
// meet in warp 0, which posts the CTA's winner; after one cluster barrier
// every warp reduces the C CTA winners.  `better` is a total order, so every
// warp of every CTA gets the same winner.
__device__ __forceinline__ RacePart race_reduce(cg::cluster_group& cluster, Smem& sm, RacePart p,
                                                int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float bw = p.w, bE = p.E;
  int bidx = p.idx;
  warp_race(bw, bE, bidx);
  if (lane == 0) sm.rpart[slot][warp] = {bw, bE, bidx};
  __syncthreads();
  if (warp == 0) {
    RacePart o = lane < kWarps ? sm.rpart[slot][lane] : RacePart{0.0f, 1.0f, 0x7FFFFFFF};
    warp_race(o.w, o.E, o.idx);
    if (lane == 0) sm.crpart[slot] = o;
  }
  cluster.sync();
  RacePart o = lane < (int)cluster.num_blocks() ? cluster.map_shared_rank(&sm, lane)->crpart[slot]
                                                : RacePart{0.0f, 1.0f, 0x7FFFFFFF};
  warp_race(o.w, o.E, o.idx);
  return o;
}

// Debug output: normalised probabilities of this thread's groups.
template <int EB, bool PROBS>
__device__ __noinline__ void write_probs(float* out, const char* s, const SliceIter& it,
                                         const RowP& r) {
#pragma unroll 1
  for (int blk = 0; blk < it.nblk; ++blk) {
    const int x = it.x(blk);
    if (x >= it.x1) break;
    Grp<EB> g;
    lds_group<EB, PROBS>(g, s, it.x0, x, it.x1);
#pragma unroll
    for (int e = 0; e < kGroup; ++e)
      if (x + e < it.x1) out[x + e] = prob<EB, PROBS>(gval<EB>(g, e), r);
  }
}

// ---------------------------------------------------------------------------
// Repetition penalty (CTRL's rule): a positive logit is divided by theta, any
// other multiplied, in fp32 round-to-nearest; a bf16 row keeps the result
// rounded to bf16, ties to even.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool theta_valid(float th) { return th > 0.0f && th <= FLT_MAX; }

template <int EB>
__device__ __forceinline__ float penalised(float l, float th) {
  float v = l > 0.0f ? __fdiv_rn(l, th) : __fmul_rn(l, th);
  if constexpr (EB == 2) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
    v = __uint_as_float((uint32_t)h << 16);
  }
  return v;
}

template <int EB>
__device__ __forceinline__ void penalise_elem(char* s, int e, float th) {
  if constexpr (EB == 2) {
    uint16_t* p = reinterpret_cast<uint16_t*>(s) + e;
    *p = (uint16_t)(__float_as_uint(penalised<2>(__uint_as_float((uint32_t)*p << 16), th)) >> 16);
  } else {
    float* p = reinterpret_cast<float*>(s) + e;
    *p = penalised<4>(*p, th);
  }
}

// ---------------------------------------------------------------------------
// Tickets.  Rows are handed out in (position, request) order by a counter in
// the workspace.  The control warp of a cluster (rank 0, last warp) takes the
// next ticket while the current row's loads are in flight, checks it, and
// loads the parameters of the row it names into sm.tk[slot]; every CTA reads
// them from there over DSMEM.
// ---------------------------------------------------------------------------
template <int EBT, int EBD>
__device__ void settle_ticket(const KParams& P, Smem& sm, int t, int slot, uint32_t tag) {
  const int lane = threadIdx.x & 31;
  Ticket tk = {0, kDone, 0, 0, 0, 0u, 0.0f, 1.0f, 0.0f, 0.0f, -1, 0, 1.0f, 0};
  t = __shfl_sync(0xffffffffu, t, 0);
  while (t < P.n_tickets) {
    const int i = t / P.B, b = t - i * P.B;
    const int kb = P.k ? P.k[b] : P.kmax;
    const int cap = P.max_new ? P.max_new[b] : 0x7FFFFFFF;
    // with a cap c <= k only rows 0 .. c-1 matter (accepting row c-1 ends the walk)
    const int last = cap <= kb ? cap - 1 : kb;
    bool take = true;
    if (kb < 0 || kb > P.kmax || cap < 1) {  // bad k or cap end the request once, at row 0
      if (i == 0 && lane == 0) write_bad_outputs(P, b, SV_ST_BAD_INPUT);
      take = false;
    } else if (i > last) {
      take = false;
    } else if (!(P.flags & SV_FLAG_NO_SKIP) && i > 0 && warp_earlier_rejected(P, b, i, tag)) {
      if (lane == 0) {
        st_relaxed(P.row_state + (size_t)b * (P.kmax + 1) + i, tag | SV_ROW_SKIPPED);
        if (P.debug) P.debug[(size_t)b * (P.kmax + 1) + i].state = SV_ROW_SKIPPED;
      }
      take = false;
    }
    if (take) {
      const bool has_d = i < kb;
      float T = 0.0f, tp = 1.0f;
      int y = 0, sl = 0;
      uint32_t rid = (uint32_t)b;
      if (lane == 0) T = P.temperature[b];  // one parameter per lane: one round trip
      if (lane == 1 && P.top_p) tp = P.top_p[b];
      if (lane == 2 && has_d) y = P.tokens[(size_t)b * P.kmax + i];
      if (lane == 3 && P.seq_len) sl = P.seq_len[b];
      if (lane == 4 && P.request_id) rid = P.request_id[b];
      float th = 1.0f;
      if (lane == 5 && P.rep_penalty) th = P.rep_penalty[b];
      th = __shfl_sync(0xffffffffu, th, 5);
      int tkk = 0;
      if (lane == 6 && P.top_k) tkk = P.top_k[b];
      tkk = __shfl_sync(0xffffffffu, tkk, 6);
      T = __shfl_sync(0xffffffffu, T, 0);
      tp = __shfl_sync(0xffffffffu, tp, 1);
      y = __shfl_sync(0xffffffffu, y, 2);
      sl = __shfl_sync(0xffffffffu, sl, 3);
      rid = __shfl_sync(0xffffffffu, rid, 4);
      float vt = 0.0f, vd = 0.0f;  // the accept-test operands
      if (has_d && y >= 0 && y < P.V) {
        const char* trow = P.target + ((size_t)b * (P.kmax + 1) + i) * P.t_ld * EBT;
        const char* drow = P.draft + ((size_t)b * P.kmax + i) * P.d_ld * EBD;
        if (lane == 0)
          vt = EBT == 2 ? __uint_as_float((uint32_t)((const uint16_t*)trow)[y] << 16)
                        : ((const float*)trow)[y];
        if (lane == 1)
          vd = EBD == 2 ? __uint_as_float((uint32_t)((const uint16_t*)drow)[y] << 16)
                        : ((const float*)drow)[y];
      }
      vt = __shfl_sync(0xffffffffu, vt, 0);
      vd = __shfl_sync(0xffffffffu, vd, 1);
      if (th != 1.0f && theta_valid(th) && has_d && y >= 0 && y < P.V) {
        // is y in row i's penalised set (the history and the drafts before i)?
        bool hit = false;
        const int32_t* h = P.rep_tokens + (size_t)b * P.rep_ld;
        for (int j = lane; j < P.rep_ld; j += 32) hit |= h[j] == y;
        for (int j = lane; j < i; j += 32) hit |= P.tokens[(size_t)b * P.kmax + j] == y;
        if (__any_sync(0xffffffffu, hit)) {
          vt = penalised<EBT>(vt, th);
          if (P.rep_draft) vd = penalised<EBD>(vd, th);
        }
      }
      const int eos = P.eos ? P.eos[b] : -1;
      tk = {t, kWork, kb, y, sl + 1 + i, rid, T, tp, vt, vd, eos < 0 ? -1 : eos, cap <= kb && i == cap - 1,
            th, tkk};
      break;
    }
    int nt = 0;
    if (lane == 0) nt = (int)atomicAdd(P.hdr + kHdrTicket, 1u);
    t = __shfl_sync(0xffffffffu, nt, 0);
  }
  tk.t = t;
  if (lane == 0) sm.tk[slot] = tk;
  __syncwarp();
}

// Just before the row that holds it starts: a row whose request has meanwhile
// seen a rejection is marked skipped and replaced by the next useful ticket.
template <int EBT, int EBD>
__device__ void recheck_ticket(const KParams& P, Smem& sm, int slot, uint32_t tag) {
  const Ticket tk = sm.tk[slot];
  if (tk.kind != kWork || (P.flags & SV_FLAG_NO_SKIP)) return;
  const int i = tk.t / P.B, b = tk.t - i * P.B;
  if (i == 0 || !warp_earlier_rejected(P, b, i, tag)) return;
  int nt = 0;
  if ((threadIdx.x & 31) == 0) {
    st_relaxed(P.row_state + (size_t)b * (P.kmax + 1) + i, tag | SV_ROW_SKIPPED);
    if (P.debug) P.debug[(size_t)b * (P.kmax + 1) + i].state = SV_ROW_SKIPPED;
    nt = (int)atomicAdd(P.hdr + kHdrTicket, 1u);
  }
  settle_ticket<EBT, EBD>(P, sm, nt, slot, tag);
}

// Is every earlier row of request b accepted?  Returns 1 (yes: this row
// decides the request), 0 (an earlier row was not accepted) or 2 (the wait
// gave up).  Warp-uniform polling: lanes read rows lane and lane + 32.
__device__ __forceinline__ int warp_wait_earlier(const KParams& P, int b, int i, uint32_t tag,
                                                 bool& qzero_seen) {
  const uint32_t* rs = P.row_state + (size_t)b * (P.kmax + 1);
  const int lane = threadIdx.x & 31;
  const uint32_t done = tag | SV_ROW_ACCEPTED;
  for (int spins = 0;; ++spins) {
    const uint32_t w0 = lane < i ? ld_relaxed(rs + lane) : done;
    const uint32_t w1 = lane + 32 < i ? ld_relaxed(rs + lane + 32) : done;
    const bool d0 = (w0 & ~0xFu) == tag && (w0 & kStateMask) != 0;
    const bool d1 = (w1 & ~0xFu) == tag && (w1 & kStateMask) != 0;
    const bool n0 = d0 && (w0 & kStateMask) != SV_ROW_ACCEPTED;
    const bool n1 = d1 && (w1 & kStateMask) != SV_ROW_ACCEPTED;
    if (__any_sync(0xffffffffu, n0 || n1)) return 0;
    if (__all_sync(0xffffffffu, d0 && d1)) {
      qzero_seen = __any_sync(0xffffffffu, ((w0 | w1) & kQZeroBit) != 0u);
      return 1;
    }
    if (spins >= P.spin_limit) return 2;
    __nanosleep(spins < 16 ? 32 : 256);
  }
}

// ---------------------------------------------------------------------------
// The kernel.  A persistent grid of clusters; each cluster works one row
// (target row i and draft row i of request b) at a time, every CTA on its
// slice of both rows in shared memory.
// ---------------------------------------------------------------------------
// Two CTAs per SM (128 registers, no spills) rather than three (80 registers,
// spills in the row loop): fewer clusters, but each row's phases run faster.
template <int EBT, int EBD, bool PROBS, bool TOPK>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const KParams P) {
  // Launched as a programmatic dependent (spec_verify), this grid may start
  // while the previous kernel (the lookahead reserve, or the previous call)
  // still runs: wait for it before anything at all is read, the workspace's
  // epoch included.  A programmatically dependent kernel that follows (the
  // commit) may then be scheduled, on an SM this grid leaves free; it reads
  // nothing of this call before its own griddepcontrol.wait.
  pdl_wait();
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ Smem sm;
  extern __shared__ __align__(128) char dyn[];
  char* s_t = dyn;              // target slice
  char* s_d = dyn + P.d_off;    // draft slice
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t epoch = *(volatile const uint32_t*)(P.hdr + kHdrEpoch);
  const uint32_t tag = epoch_tag(epoch);
  const uint32_t k0 = P.seed_lo, k1 = P.seed_hi;
  const bool lead = rank == 0 && tid == 0;                // publishes states and outputs
  const bool ctl = rank == 0 && warp == kWarps - 1;       // takes tickets, resolves
  uint32_t phase_t = 0u, phase_d = 0u;  // mbarrier parities

  if (tid == 0) {
    mbar_init(&sm.bar[0]), mbar_init(&sm.bar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (ctl) {
    int t0 = 0;
    if (lane == 0) t0 = (int)atomicAdd(P.hdr + kHdrTicket, 1u);
    settle_ticket<EBT, EBD>(P, sm, t0, 0, tag);
  }
  cluster.sync();
  for (int iter = 0;; ++iter) {
    const int parity = iter & 1;
    const Ticket tk = cluster.map_shared_rank(&sm, 0)->tk[parity];
    if (tk.kind == kDone) break;

    // ---------------------------------------------------------------- row setup
    const int t = tk.t;
    const int i = t / P.B, b = t - i * P.B;
    const bool has_d = i < tk.kb;
    const size_t row_t = (size_t)b * (P.kmax + 1) + i;
    const size_t row_d = (size_t)b * P.kmax + i;
    SliceIter it;
    it.x0 = rank * P.slice;
    it.x1 = min(P.V, it.x0 + P.slice);
    it.nblk = it.x1 > it.x0 ? (it.x1 - it.x0 + kBlk - 1) / kBlk : 0;
    it.V = P.V;
    it.stride = kBlk, it.tid = (int)threadIdx.x;

    // ------------------------------------ TMA: this CTA's slice of both rows
    if (tid == 0) {
      const char* trow = P.target + row_t * P.t_ld * EBT;
      const char* drow = P.draft + row_d * P.d_ld * EBD;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // prior reads before new writes
      // one copy per row: the TMA unit's cost grows with the number of
      // copies far more than with their size
      if (it.nblk > 0) {
        const uint32_t bt = (uint32_t)(((it.x1 - it.x0) * EBT + 15) & ~15);
        mbar_expect_tx(&sm.bar[0], bt);
        bulk_g2s(s_t, trow + (size_t)it.x0 * EBT, bt, &sm.bar[0]);
        if (has_d) {
          const uint32_t bd = (uint32_t)(((it.x1 - it.x0) * EBD + 15) & ~15);
          mbar_expect_tx(&sm.bar[1], bd);
          bulk_g2s(s_d, drow + (size_t)it.x0 * EBD, bd, &sm.bar[1]);
        }
      }
    }

    // repetition penalty: mark this slice's penalised elements in a bitmap
    // (one bit per element, so that a token listed twice counts once) while
    // the slices load; they are rewritten once the loads have landed
    const float theta = tk.theta;
    const bool rep = theta != 1.0f && theta_valid(theta) && it.nblk > 0;
    uint32_t* rmask = reinterpret_cast<uint32_t*>(&sm.wb);
    if (rep) {
      for (int j = tid; j < kMaxBlk * kBlk / 32; j += kThreads) rmask[j] = 0u;
      __syncthreads();
      const int32_t* h = P.rep_tokens + (size_t)b * P.rep_ld;
      const int32_t* dt = P.tokens + (size_t)b * P.kmax;
      for (int j = tid; j < P.rep_ld + i; j += kThreads) {
        const int x = j < P.rep_ld ? h[j] : dt[j - P.rep_ld];
        if (x >= it.x0 && x < it.x1)
          atomicOr(&rmask[(x - it.x0) >> 5], 1u << ((x - it.x0) & 31));
      }
    }

    const float T = tk.T, top_p = tk.top_p;
    const int y = tk.y, pos = tk.pos;
    const uint32_t rid = tk.rid;
    // the accept uniform depends only on (seed, position, request): draw it
    // while the slices load
    const float u_row = uniform_from_bits(philox4x32_10(make_uint4(0u, (uint32_t)pos, rid, 1u), k0, k1).x);
    const bool params_ok = (T >= 0.0f) && (T <= FLT_MAX) && (top_p > 0.0f) && (top_p <= 1.0f) &&
                           theta_valid(theta);
    const bool y_ok = !has_d || (y >= 0 && y < P.V);
    const bool greedy = T == 0.0f;
    RowP rt, rd;
    rt.greedy = rd.greedy = greedy;
    rt.c = greedy ? 0.0f : kLog2e / T;
    rt.invT = rd.invT = greedy ? 0.0f : 1.0f / T;
    rd.c = PROBS ? 1.0f : rt.c;
    rt.Dstar = rd.Dstar = kNoFilter;

    // --------------------------------------------- sweep 1: raw maxima
    uint32_t mt2 = 0xFF80FF80u, md2 = 0xFF80FF80u;
    float rmt = -INFINITY, rmd = PROBS ? 0.0f : -INFINITY;
    bool landed = true;
    if (it.nblk > 0) {
      landed &= mbar_wait(&sm.bar[0], phase_t, P.err);
      if (has_d) landed &= mbar_wait(&sm.bar[1], phase_d, P.err);
      phase_t ^= 1u;
      if (has_d) phase_d ^= 1u;
    }
    if (rep) {
      __syncthreads();  // the bitmap is complete
      const bool pen_d = has_d && P.rep_draft;
      for (int w = tid; w < (it.x1 - it.x0 + 31) >> 5; w += kThreads) {
        for (uint32_t m = rmask[w]; m; m &= m - 1u) {
          const int e = (w << 5) + __ffs(m) - 1;
          penalise_elem<EBT>(s_t, e, theta);
          if (pen_d) penalise_elem<EBD>(s_d, e, theta);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int blk = 0; blk < kMaxBlk; ++blk) {
      const int x = it.x(blk);
      if (blk < it.nblk && x < it.x1) {
        Grp<EBT> g;
        lds_group<EBT, false>(g, s_t, it.x0, x, it.x1);
        max_group<EBT>(g, mt2, rmt);
        if (has_d) {
          Grp<EBD> h;
          lds_group<EBD, PROBS>(h, s_d, it.x0, x, it.x1);
          max_group<EBD>(h, md2, rmd);
        }
      }
    }
    rmt = max_value<EBT>(mt2, rmt);
    rmd = max_value<EBD>(md2, rmd);
    // this thread's maxima in the weight domain
    const float mt = rmt;
    const float md = (PROBS && !greedy) ? (rmd > 0.0f ? lg2(rmd) * rd.invT : -INFINITY) : rmd;
    // bf16 logit rows with top_p < 1 count their top-p window during sweep 2
    // top-k (0 < top_k < V) runs before top-p; its rows count no prebuilt
    // top-p window (the top-p target depends on the top-k mass)
    const bool topk = TOPK && !greedy && params_ok && tk.top_k > 0 && tk.top_k < P.V;
    const bool topp = !greedy && top_p < 1.0f && params_ok && !topk;
    const bool win_t = EBT == 2 && topp;
    const bool win_d = EBD == 2 && !PROBS && topp && has_d;
    if (win_t || win_d)
      for (int j = tid; j < 512; j += kThreads) (&sm.hist[0][0][0])[j] = 0u;

    // ------ exchange 1: row maxima, and a lower bound of the weight sums
    // Every thread's own maximum weighs 1 relative to itself, so the sum over
    // threads of 2^((m_thread - M) c) is at most the row's weight sum S.
    {
      float Mw = mt, Lw = mt == -INFINITY ? 0.0f : 1.0f;
      float Nw = md, Kw = md == -INFINITY ? 0.0f : 1.0f;
      warp_ms(Mw, Lw, rt.c, greedy);
      warp_ms(Nw, Kw, rd.c, greedy);
      float Rw = rmd;
#pragma unroll
      for (int o = 16; o; o >>= 1) Rw = fmaxf(Rw, __shfl_xor_sync(0xffffffffu, Rw, o));
      const bool warp_bad = __any_sync(0xffffffffu, !landed);
      if (lane == 0)
        sm.part[warp] = {make_float4(Mw, Lw, Rw, warp_bad ? 1.0f : 0.0f), make_float4(Nw, Kw, 0.0f, 0.0f)};
    }
    __syncthreads();
    if (warp == 0) {  // the CTA's partial
      const StatPart c = combine_parts(lane < kWarps ? sm.part[lane] : neutral_part<PROBS>(), rt.c,
                                       rd.c, greedy);
      if (lane == 0) sm.cpart = c;
    }
    cluster.sync();  // partials visible cluster-wide
    float St_lb, Sd_lb;
    bool slice_bad;
    {
      const StatPart c = combine_parts(
          lane < C ? cluster.map_shared_rank(&sm, lane)->cpart : neutral_part<PROBS>(), rt.c, rd.c, greedy);
      rt.m = rt.mz = c.a.x;
      rd.m = c.a.z;   // raw maximum (logit or probability): defines the top-p keys
      rd.mz = c.d.x;  // maximum in the weight domain (== raw max except probabilities, T > 0)
      St_lb = c.a.y, Sd_lb = c.d.y;
      slice_bad = c.a.w != 0.0f;
    }
    rt.kmax = vkey<EBT>(rt.m);
    rd.kmax = vkey<EBD>(rd.m);

    // window floors from the lower bound of S (a lower floor than S gives)
    uint32_t thr2_t = 0x7FFF7FFFu, thr2_d = 0x7FFF7FFFu;  // NaN pairs: nothing passes
    const int nguess = min(P.V, kWindowGuess);
    if (win_t) {
      RowP q = rt;
      q.S = St_lb;
      thr2_t = bf16_pair_of(vkey_value<2>(window_lo_key(q, top_p, nguess)));
    }
    if (win_d) {
      RowP q = rd;
      q.S = Sd_lb;
      thr2_d = bf16_pair_of(vkey_value<2>(window_lo_key(q, top_p, nguess)));
    }

    // ------------- sweep 2: weight sums to the row maxima, window candidates
    float st = 0.0f, sd = 0.0f;
    uint32_t wt_lo = 0u, wt_hi = 0u, wd_lo = 0u, wd_hi = 0u;
    int wt_n = 0, wd_n = 0;
#pragma unroll 2
    for (int blk = 0; blk < it.nblk; ++blk) {
      const int x = it.x(blk);
      if (x < it.x1) {
        Grp<EBT> g;
        lds_group<EBT, false>(g, s_t, it.x0, x, it.x1);
        st += sum_group<EBT, false>(g, greedy, rt.mz, rt.c, rt.invT);
        if constexpr (EBT == 2) {
          if (win_t) {
            const uint32_t m = window_bits_bf16(make_uint4(g.w[0], g.w[1], g.w[2], g.w[3]), thr2_t, x, it.x1);
            wt_n += __popc(m);
            if (blk < 4) wt_lo |= m << (8 * blk);
            else wt_hi |= m << (8 * (blk - 4));
          }
        }
        if (has_d) {
          Grp<EBD> h;
          lds_group<EBD, PROBS>(h, s_d, it.x0, x, it.x1);
          sd += sum_group<EBD, PROBS>(h, greedy, rd.mz, rd.c, rd.invT);
          if constexpr (EBD == 2 && !PROBS) {
            if (win_d) {
              const uint32_t m = window_bits_bf16(make_uint4(h.w[0], h.w[1], h.w[2], h.w[3]), thr2_d, x, it.x1);
              wd_n += __popc(m);
              if (blk < 4) wd_lo |= m << (8 * blk);
              else wd_hi |= m << (8 * (blk - 4));
            }
          }
        }
      }
    }
    if constexpr (EBT == 2) {
      if (win_t) window_commit_bf16(s_t, rt.kmax, wt_lo, wt_hi, wt_n, it, sm.hist[0][0], sm.wb.bin[warp]);
    }
    if constexpr (EBD == 2 && !PROBS) {
      if (win_d) window_commit_bf16(s_d, rd.kmax, wd_lo, wd_hi, wd_n, it, sm.hist[0][1], sm.wb.bin[warp]);
    }

    // ------ exchange 2: the weight sums (and the window histograms with them)
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      st += __shfl_xor_sync(0xffffffffu, st, o);
      sd += __shfl_xor_sync(0xffffffffu, sd, o);
    }
    if (lane == 0) sm.spart[warp] = make_float2(st, sd);
    __syncthreads();
    if (warp == 0) {  // the CTA's sums, warps in order
      float2 v = lane < kWarps ? sm.spart[lane] : make_float2(0.0f, 0.0f);
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
      }
      if (lane == 0) sm.cspart = v;
    }
    cluster.sync();
    {
      float2 v = lane < C ? cluster.map_shared_rank(&sm, lane)->cspart : make_float2(0.0f, 0.0f);
      float a = v.x, c2 = v.y;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        c2 += __shfl_xor_sync(0xffffffffu, c2, o);
      }
      rt.S = a, rd.S = c2;
      if (slice_bad) rt.S = __int_as_float(0x7FC00000);  // a slice never landed: the row is invalid
    }
    rt.Z = rt.S, rd.Z = rd.S;
    rt.invZ = 1.0f / rt.Z, rd.invZ = 1.0f / rd.Z;
    rt.vstar = -INFINITY;
    rd.vstar = PROBS ? 0.0f : -INFINITY;

    // NaN / +inf inputs surface as a non-finite sum or maximum
    const bool bad_t = !(rt.S >= 1.0f && rt.S <= FLT_MAX) || !(rt.m <= FLT_MAX) ||
                       rt.m == -INFINITY;
    const bool bad_d = has_d && (!(rd.S >= 1.0f && rd.S <= FLT_MAX) || !(rd.m <= FLT_MAX) ||
                                 (PROBS ? !(rd.m > 0.0f) : rd.m == -INFINITY));
    const bool row_bad = bad_t || bad_d || !params_ok || !y_ok;

    // The next ticket: taken by the control warp while warps 0 and 1 resolve
    // the top-p boundary (the CTA's other warps wait for them anyway).
    if (ctl) {
      int nt = 0;
      if (lane == 0) nt = (int)atomicAdd(P.hdr + kHdrTicket, 1u);
      settle_ticket<EBT, EBD>(P, sm, nt, parity ^ 1, tag);
    }

    // ---------------------------------------------------------------- top-p
    if (!row_bad && (topk || (!greedy && top_p < 1.0f)))
      filter_rows<EBT, EBD, PROBS>(cluster, sm, s_t, s_d, it, has_d, top_p, topk ? tk.top_k : 0, rt, rd,
                                   win_t, win_d);

    // ---------------------------------------------------------- accept test
    // Every CTA evaluates the test identically from the same values.
    int state;
    bool qzero = false;
    float p_y = 0.0f, q_y = 0.0f, u = 0.0f;
    if (row_bad) {
      state = SV_ROW_INVALID;
    } else if (has_d) {
      p_y = prob<EBT, false>(tk.vt, rt);
      q_y = prob<EBD, PROBS>(tk.vd, rd);
      u = u_row;
      qzero = q_y == 0.0f;
      state = (u * q_y < p_y) ? SV_ROW_ACCEPTED : SV_ROW_REJECTED;
      // an accepted EOS id, or the last row the output cap allows, ends the request
      if (state == SV_ROW_ACCEPTED && ((tk.eos >= 0 && y == tk.eos) || tk.cap_row))
        state = SV_ROW_TERMINAL;
    } else {
      state = SV_ROW_BONUS;
    }
    if (lead && !((P.flags & SV_FLAG_TEST_WITHHOLD) && row_t == 0)) {
      st_relaxed(P.row_state + row_t, tag | (qzero ? kQZeroBit : 0u) | (uint32_t)state);
      if (P.debug) {
        sv_row_debug d;
        d.p_y = p_y, d.q_y = q_y, d.u = u;
        d.p_kept = greedy || rt.Dstar == kNoFilter ? 1.0f : rt.Z / rt.S;
        d.q_kept = !has_d || greedy || rd.Dstar == kNoFilter ? 1.0f : rd.Z / rd.S;
        d.state = state;
        d.p_thr_key = rt.Dstar == kNoFilter ? -1 : (int32_t)(rt.kmax - rt.Dstar);
        d.q_thr_key = (!has_d || rd.Dstar == kNoFilter) ? -1 : (int32_t)(rd.kmax - rd.Dstar);
        P.debug[row_t] = d;
      }
    }

    // -------------------------------------------------- debug: normalised rows
    if (P.probs_p && !row_bad) write_probs<EBT, false>(P.probs_p + row_t * (size_t)P.V, s_t, it, rt);
    if (P.probs_q && has_d && !row_bad)
      write_probs<EBD, PROBS>(P.probs_q + row_d * (size_t)P.V, s_d, it, rd);

    // --------------------------------------------- resolve: is this row the one?
    bool ended = false;  // a barrier after the re-check has published the next ticket
    if (state != SV_ROW_ACCEPTED) {
      if (ctl) {
        bool qz = false;
        int resolver = warp_wait_earlier(P, b, i, tag, qz);
        if (lane == 0) {
          if (resolver == 2) {
            report(P.err, SV_ERR_TIMEOUT);
            write_bad_outputs(P, b, SV_ST_TIMEOUT);
            resolver = 0;
          } else if (resolver == 1 && state == SV_ROW_INVALID) {
            write_bad_outputs(P, b, SV_ST_BAD_INPUT);
            resolver = 0;
          }
          sm.decide[0] = resolver;
          sm.decide[1] = (int)((qzero || qz) ? SV_ST_Q_ZERO : 0u);
        }
        // the next row may have become skippable meanwhile; the barrier
        // below publishes both the decision and the next ticket
        recheck_ticket<EBT, EBD>(P, sm, parity ^ 1, tag);
      }
      cluster.sync();
      ended = true;
      const int* dc = cluster.map_shared_rank(&sm.decide[0], 0);
      const int resolver = dc[0];
      const uint32_t st_bits = (uint32_t)dc[1];
      if (resolver && state == SV_ROW_TERMINAL) {
        // the accepted drafts 0 .. i are the whole output: no correction or bonus
        if (lead) {
          int32_t* ot2 = P.out_tokens + (size_t)b * (P.kmax + 1);
          for (int j = 0; j <= i; ++j) ot2[j] = P.tokens[(size_t)b * P.kmax + j];
          for (int j = i + 1; j <= P.kmax; ++j) ot2[j] = -1;
          P.accepted[b] = i + 1;
          P.num_emitted[b] = i + 1;
          P.status[b] = st_bits | ((tk.eos >= 0 && y == tk.eos) ? SV_ST_EOS : SV_ST_CAPPED);
        }
      } else if (resolver) {
        const bool residual = state == SV_ROW_REJECTED;
        RacePart best = {0.0f, 1.0f, 0x7FFFFFFF};
        race_slice<EBT, EBD, PROBS>(s_t, s_d, it, residual, rt, rd, (uint32_t)pos, rid, k0, k1,
                                    sm.wb.idx[warp], best);
        RacePart win = race_reduce(cluster, sm, best, 0);
        uint32_t extra = 0u;
        if (!(win.w > 0.0f)) {
          // residual numerically empty: draw from p with the same exponentials
          extra = SV_ST_RESIDUAL_EMPTY;
          best = {0.0f, 1.0f, 0x7FFFFFFF};
          race_slice<EBT, EBD, PROBS>(s_t, s_d, it, false, rt, rd, (uint32_t)pos, rid, k0, k1,
                                      sm.wb.idx[warp], best);
          win = race_reduce(cluster, sm, best, 1);
        }
        if (lead) {
          int32_t* ot2 = P.out_tokens + (size_t)b * (P.kmax + 1);
          for (int j = 0; j < i; ++j) ot2[j] = P.tokens[(size_t)b * P.kmax + j];
          ot2[i] = win.idx;
          for (int j = i + 1; j <= P.kmax; ++j) ot2[j] = -1;
          P.accepted[b] = i;
          P.num_emitted[b] = i + 1;
          P.status[b] = st_bits | extra;
        }
      }
    }

    if (!ended) {
      // the next row may have become skippable meanwhile; the end-of-row
      // barrier then publishes its ticket
      if (ctl) recheck_ticket<EBT, EBD>(P, sm, parity ^ 1, tag);
      cluster.sync();
    }
  }

  // all peers must be done reading rank 0's shared memory before it exits
  cluster.sync();
  if (lead) {
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
// The _topk variants also run the top-k filter; the others never do (the
// filter's code in the row loop costs the plain variants about 2% of their
// time, so a call without top_k runs a variant without it).
KernelFn kernel_bf16_bf16_logits();
KernelFn kernel_bf16_f32_probs();
KernelFn kernel_bf16_f32_logits();
KernelFn kernel_f32_f32_logits();
KernelFn kernel_f32_f32_probs();
KernelFn kernel_f32_bf16_logits();
KernelFn kernel_bf16_bf16_logits_topk();
KernelFn kernel_bf16_f32_probs_topk();
KernelFn kernel_bf16_f32_logits_topk();
KernelFn kernel_f32_f32_logits_topk();
KernelFn kernel_f32_f32_probs_topk();
KernelFn kernel_f32_bf16_logits_topk();

size_t workspace_bytes_for(int B, int kmax);

}  // namespace sv
