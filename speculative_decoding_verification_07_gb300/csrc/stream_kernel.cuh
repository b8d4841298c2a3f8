#pragma once
// Streaming verification kernel (device code).  Same method and results as
// verify_kernel.cuh ("Speculative decoding: accelerate LLM generation without
// changing its answers", sections 2-4: the transformed p_i and q_i, accept
// y_i iff u_i q_i(y_i) < p_i(y_i) left to right, the correction from
// normalize(max(0, p - q)) at the first rejection or the bonus token from
// p_{k_b}, both drawn by an exponential race), laid out so that HBM streams
// at full rate.
//
// GB300 design
//  * One persistent CTA per SM with three roles: a producer warp, two groups
//    of eight consumer warps and three finisher warps.  The producer takes
//    work tickets from counters in the workspace and pulls each item into a
//    ring of shared-memory stages with 1-D TMA bulk copies (cp.async.bulk,
//    one mbarrier per stage); item n goes to consumer group n % 2, so while
//    one group waits at a barrier or on latency the other computes.  The
//    consumers hand each stage back through an "empty" mbarrier and pass
//    their results to the finishers through a small shared-memory ring; the
//    finishers do everything that waits on global memory (partials, arrival
//    counters, merges, the request resolution), so the consumers only
//    compute.  No CTA ever waits on another CTA's shared memory.
//  * Three kinds of items, all one vocabulary chunk of one row pair (target
//    row i and, for i < k_b, draft row i of request b):
//      - row items (first pass, static tickets in (position, request, chunk)
//        order): the chunk's maxima and weight sums relative to them;
//      - window items (bf16 logit rows with top_p < 1): once the first pass
//        of a row pair is merged its maxima are exact, and each chunk is read
//        again (from L2) to count the bf16 values in a band of at most 256
//        keys just below them; a boundary below the band asks for the next
//        band down;
//      - race items: the exponential race of a resolved request's rejection
//        or bonus row over that chunk.
//    Window and race items come from a queue of slots that the producers
//    serve before any static ticket, so the rows on the critical path move
//    first.  Rows of a request behind a known rejection are never loaded.
//  * The finisher that completes a row pair's first pass merges the chunk
//    partials; without top-p it runs the accept test at once, else it queues
//    the window.  The finisher that completes the window finds the top-p
//    boundaries, runs the accept test and publishes the decision in the
//    request's state words.  Whoever completes "rows 0..f-1 accepted, row f
//    not" resolves the request: a rejection or bonus row queues the race, and
//    the last race item writes the request's outputs.
//  * Per-call state lives in two halves of the workspace used on alternate
//    calls: each call zeroes the half the next call will use.
#include "verify_kernel.cuh"

namespace sv {
namespace stream {

constexpr int kNG = 2;               // consumer groups, each on its own items
constexpr int kGW = 8;               // warps per consumer group
constexpr int kGT = kGW * 32;        // threads per consumer group
constexpr int kCW = kNG * kGW;       // consumer warps (warps 0-15; group g: warps 8g .. 8g+7)
constexpr int kProducerWarp = kCW;   // warp 16
constexpr int kFinisherWarp = kCW + 1;  // warps 17 .. 17 + kFW - 1
constexpr int kFW = 3;               // finisher warps; hand-off slot f goes to finisher f % kFW
constexpr int kAllThreads = kCW * 32 + 32 + 32 * kFW;
constexpr int kNF = 6;               // finisher hand-off slots; item n uses slot n % kNF
static_assert(kNF % kFW == 0 && kNF % kNG == 0, "slots split evenly over finishers and groups");
static_assert(kNF / kNG >= kFW, "each group's slots reach every finisher");
constexpr int kBins = 256;
constexpr int kMaxNs = 6;
constexpr int kMaxChunks = 32;
constexpr uint32_t kNA = 1024u;      // request word na = kNA - first non-accepted row (0: none)
constexpr float kDepthMargin = 1.0f; // log2 units added to the deepest nucleus seen
// Tuning: unroll of the consumers' group loops (the code must stay small
// enough for the instruction cache) and the window depth, in log2 units of
// the weight, used before any nucleus of the call has been measured (0: the
// full 256-key window).
#ifndef SV_STREAM_UNROLL
#define SV_STREAM_UNROLL 8
#endif
#ifndef SV_STREAM_DEPTH0
#define SV_STREAM_DEPTH0 0.0f
#endif
constexpr int kStreamUnroll = SV_STREAM_UNROLL;

// Items are one chunk of a row pair: 32 KB of stage for every dtype mix.
template <int EBT, int EBD>
__host__ __device__ constexpr int chunk_elems() {
  return (EBT == 2 && EBD == 2) ? 8192 : 4096;
}
template <int EBT, int EBD>
__host__ __device__ constexpr int stage_bytes() {
  return chunk_elems<EBT, EBD>() * (EBT + EBD);
}
// Item n uses stage n % NS; a multiple of kNG, so each group has its own stages.
template <int EBT, int EBD>
__host__ __device__ constexpr int num_stages() {
  return 6;
}
static_assert(6 % kNG == 0 && 6 <= kMaxNs, "stages split evenly over the groups");

enum : int { kEnd = 0, kRowItem = 1, kRaceItem = 2, kBadItem = 3, kWinItem = 4 };
enum : int { kRaceResidual = 1, kRaceBonus = 2, kWindowSlot = 3 };  // queue slot kinds

// ---------------------------------------------------------------------------
// Workspace records
// ---------------------------------------------------------------------------
struct Hdr {            // fixed words at byte 64 of the workspace header
  uint32_t parity;      // which state half this call uses
  uint32_t ticket;      // next static ticket (row items)
  uint32_t exit_cnt;    // CTAs finished
  uint32_t dticket;     // next queued ticket (window and race items: slot * n_ch + chunk)
  uint32_t depth_t;     // deepest nuclei of the previous call (log2 units, float bits):
  uint32_t depth_d;     // the first bands of a call start from them
  uint32_t pad[10];
};

struct CallSt {         // per call, zeroed by the previous call
  unsigned long long cnt;  // (requests resolved << 32) | queue slots claimed
  uint32_t n_done;      // requests whose outputs are written
  uint32_t depth_t;     // deepest target nucleus seen, log2 units (float bits)
  uint32_t depth_d;
  uint32_t pad[11];
};
static_assert(sizeof(CallSt) == 64, "");

// Decisions of a request.  With kmax <= kFastK one 64-bit word holds them
// all -- bit i: row i accepted; bit 21 + i: row i decided and not accepted;
// bit 42 + i: row i's test saw q(y) == 0 -- so that one atomic OR both
// publishes a decision and tells its issuer whether it completed the request
// ("rows 0 .. f-1 accepted, row f not").  Larger kmax use acc / qz / na with
// a fence-separated check and a CAS on `resolved`.
constexpr int kFastK = 20;
struct ReqSt {
  unsigned long long acc;   // bit i: row i accepted (kmax > kFastK)
  unsigned long long qz;    // bit i: row i's test saw q(y) == 0 (kmax > kFastK)
  unsigned long long best;  // race winner: (key bits << 32) | (0xFFFFFFFF - token)
  unsigned long long w;     // the single decision word (kmax <= kFastK)
  uint32_t na;              // kNA - first non-accepted row, or 0 (kmax > kFastK)
  uint32_t resolved;        // 0 -> 1 by the resolver (2: timed out)
  uint32_t race_cnt;        // race items finished
  uint32_t pad[5];
};
static_assert(sizeof(ReqSt) == 64, "");

// A queue slot: two 64-bit words, each written once per call, so that a
// reader that sees both non-zero sees the slot complete.
//   w0: bit 63 set | row << 32 | b << 8 | kind
//   w1: window: lo_t | hi_t << 16 | lo_d << 32 | hi_d << 48 (hi_t > 0)
//       race:   pos | request id << 32 (pos > 0)
struct Slot {
  unsigned long long w0, w1;
};
constexpr unsigned long long kSlotFilled = 1ull << 63;

struct PairSt {
  uint32_t arrive;      // first-pass chunks finished
  uint32_t warrive;     // window chunks finished (this band)
  uint32_t state;       // SV_ROW_* once decided
  uint32_t wside;       // bits 0/1: target/draft counted in this band; bits 8+: band index
  uint32_t lo_t, hi_t;  // the band's bf16 order keys, target
  uint32_t lo_d, hi_d;  // and draft
};
constexpr int kMaxBands = 2;  // bands per row before the exact descent takes over

// A row pair's first-pass statistics, kept for its window.
struct PairStats {
  float Mt, St, Md, Sd;  // maxima and weight sums (relative to them)
  float vt, vd;          // the values at the proposal
  float above_t, above_d;  // mass of the keys above the current band
  uint32_t y_ok;
  uint32_t pad[7];
};
static_assert(sizeof(PairStats) == 64, "");

// One side (target or draft) of a decided row: everything the race and the
// normalised-row writer need to evaluate prob(v).
struct RowSide {
  float m, mz, c, invT;
  float Z, invZ, vstar;
  uint32_t Dstar;       // kept iff vkey(m) - vkey(v) <= Dstar; kNoFilter = all
};
struct RowRec {
  RowSide t, d;
};
static_assert(sizeof(RowRec) == 64, "");

// chunk partial: (Mt, St, Md, Sd) | (vt, vd, has_y, 0) | window counts of
// the band, 2 x 256 u16 (bin j: key hi - j)
constexpr int kPartHead = 32;

// ---------------------------------------------------------------------------
// Kernel parameters
// ---------------------------------------------------------------------------
struct SParams {
  int B, kmax, V, n_ch;
  uint32_t flags;
  const char* target;
  int64_t t_ld;
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
  const int32_t* eos;
  const int32_t* max_new;
  Hdr* hdr;
  char* state[2];       // per-call state halves
  size_t state_words;   // u32 words per half
  RowRec* rows;         // [B][kmax+1]
  PairStats* pstats;    // [B][kmax+1]
  char* parts;          // [B][kmax+1][n_ch] partials
  int part_bytes;       // kPartHead, plus 2 * 512 with histograms
  int hist;             // partials carry window histograms
  uint32_t n_slots;     // queue slots: kMaxBands windows per row pair, one race per request
  int* err;
  unsigned long long slot_wait_ns;  // bound of a wait for a race slot
  uint32_t n_static;    // static tickets: (kmax + 1) * B * n_blk
  int n_blk;            // tickets per row: blocks of up to kBatch chunks
};
constexpr int kBatch = 4;  // chunks per ticket (one round trip of the producer settles them all)

// state-half layout: CallSt | ReqSt[B] | Slot[n_slots] | PairSt[B][kmax+1]
__host__ __device__ inline size_t slots_for(int B, int kmax) {
  return (size_t)B * (size_t)(kmax + 1) * kMaxBands + (size_t)B;
}
__host__ __device__ inline size_t state_bytes_for(int B, int kmax) {
  return sizeof(CallSt) + (size_t)B * sizeof(ReqSt) + slots_for(B, kmax) * sizeof(Slot) +
         (size_t)B * (size_t)(kmax + 1) * sizeof(PairSt);
}
__device__ __forceinline__ CallSt* call_st(char* s) { return reinterpret_cast<CallSt*>(s); }
__device__ __forceinline__ ReqSt* req_st(char* s, int b) {
  return reinterpret_cast<ReqSt*>(s + sizeof(CallSt)) + b;
}
__device__ __forceinline__ Slot* slot_st(char* s, int B, int q) {
  return reinterpret_cast<Slot*>(s + sizeof(CallSt) + (size_t)B * sizeof(ReqSt)) + q;
}
__device__ __forceinline__ PairSt* pair_st(char* s, const SParams& P, size_t pair) {
  return reinterpret_cast<PairSt*>(s + sizeof(CallSt) + (size_t)P.B * sizeof(ReqSt) +
                                   (size_t)P.n_slots * sizeof(Slot)) +
         pair;
}

// ---------------------------------------------------------------------------
// Shared memory
// ---------------------------------------------------------------------------
struct SHdr {           // one stage's item, written by the producer
  int kind, b, i, c;
  int x0, n, has_d, kb;
  float T, top_p;
  int race, pos;
  uint32_t rid;
  int y;                // the row's proposal (draft rows)
  int win;              // window items: bit 0 target, bit 1 draft
  uint32_t lo_t, hi_t, lo_d, hi_d;  // window items: the band's keys
  int pad;
  RowRec rr;            // race items: the decided row
};

// Consumer -> finisher hand-off of one item.
struct alignas(16) Fin {
  int kind, b, i, c;
  int has_d, kb, race, pos;
  float T, top_p;
  uint32_t rid;
  int y;
  float vt, vd;         // the values at y when y lies in this chunk
  int has_y, win;       // win: bit 0 target window, bit 1 draft window
  float rw, rE;         // race items: the chunk's winner
  int ridx, pad;
  RowRec rr;            // race items: the decided row
  float4 wp[kGW];       // row items: per consumer warp (max, sum) of target and draft
  uint32_t hist[2][kBins];  // window items: counts, bin j = key hi - j
};

struct alignas(16) SSmem {
  unsigned long long full[kMaxNs], empty[kMaxNs];
  unsigned long long fin_full[kNF], fin_empty[kNF];
  SHdr hdr[kMaxNs];
  Fin fin[kNF];
  float fh[kFW][kBins]; // finisher scratch: descent histogram
  RacePart rp[kCW];
  uint16_t wb[kCW][256];  // per consumer warp: race candidates / window groups
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
// Barrier of consumer group g (named barrier 1 + g).
__device__ __forceinline__ void gbar(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "n"(kGT) : "memory");
}

__device__ __forceinline__ void fence_sc() { asm volatile("fence.sc.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void mbar_init_n(unsigned long long* bar, int n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_arrive1(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(unsigned long long* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait (the bound is time, not a poll count): false, with
// SV_ERR_TIMEOUT reported, if the phase has not completed after `ns`.
constexpr unsigned long long kStageWaitNs = 4000000000ull;   // consumers, producer
constexpr unsigned long long kFinWaitNs = 6000000000ull;     // finishers wait on the consumers
__device__ __forceinline__ bool mbar_wait_ns(unsigned long long* bar, uint32_t parity, int* err,
                                             unsigned long long ns, uint32_t max_sleep = 256u) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  // The suspend hint of try_wait parks the warp only briefly: back off with
  // a sleep between tries, so that waiting warps leave the issue slots (and
  // the instruction cache) to the warps that have work.
  uint32_t sleep = 32u;
  for (;;) {
    __nanosleep(sleep);
    if (mbar_try_wait(bar, parity)) return true;
    if (gtimer() - t0 > ns) break;
    sleep = sleep < max_sleep ? sleep * 2u : max_sleep;
  }
  report(err, SV_ERR_TIMEOUT);
  return false;
}

// Optional event trace (built only with -DSV_TRACE): timestamped events of
// the pipeline roles, for studying where an item's time goes.  Compiled out
// otherwise.
#ifdef SV_TRACE
static __device__ unsigned long long* g_sv_trace = nullptr;
static __device__ unsigned int g_sv_trace_n = 0u, g_sv_trace_cap = 0u;  // cap: events per CTA
__device__ __forceinline__ unsigned int& trace_slot() {
  __shared__ unsigned int n;  // events recorded by this CTA
  return n;
}
__device__ __forceinline__ void trace_ev(uint32_t ev, uint32_t a, uint32_t b) {
  const unsigned idx = atomicAdd(&trace_slot(), 1u);
  if (idx < g_sv_trace_cap) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    unsigned long long* p = g_sv_trace + 2ull * ((unsigned long long)blockIdx.x * g_sv_trace_cap + idx);
    p[0] = gtimer();
    p[1] = ((unsigned long long)(ev & 0xFF) << 56) | ((unsigned long long)(smid & 0xFF) << 48) |
           ((unsigned long long)(a & 0xFFFFFF) << 24) | (b & 0xFFFFFF);
  }
}
#define SV_TR(ev, a, b) trace_ev((ev), (uint32_t)(a), (uint32_t)(b))
#else
#define SV_TR(ev, a, b) ((void)0)
#endif

// Release the stage: each warp of the consuming group arrives once after its last read.
__device__ __forceinline__ void release_stage(SSmem& sm, int s) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive1(&sm.empty[s]);
}

__device__ __forceinline__ uint32_t key16(float bf16_value) { return vkey<2>(bf16_value); }

__device__ __forceinline__ unsigned long long race_key(float w, float E, int idx) {
  const float key = w > 0.0f ? __fdiv_rn(w, E) : 0.0f;
  return ((unsigned long long)__float_as_uint(key) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ bool row_params_ok(float T, float top_p) {
  return (T >= 0.0f) && (T <= FLT_MAX) && (top_p > 0.0f) && (top_p <= 1.0f);
}

template <int EB>
__device__ __forceinline__ float row_value(const char* row, int y) {
  return EB == 2 ? __uint_as_float((uint32_t)__ldcg((const unsigned short*)row + y) << 16)
                 : __ldcg((const float*)row + y);
}

// Weight-domain maximum from the raw maximum (identical wherever it is used).
template <bool PROBS>
__device__ __forceinline__ float weight_max(float m, bool greedy, float invT) {
  if (PROBS && !greedy) return m > 0.0f ? lg2(m) * invT : -INFINITY;
  return m;
}

static __device__ void bad_outputs(const SParams& P, int b, uint32_t st) {
  P.accepted[b] = -1;
  P.num_emitted[b] = 0;
  P.status[b] = st;
  for (int j = 0; j <= P.kmax; ++j) P.out_tokens[(size_t)b * (P.kmax + 1) + j] = -1;
}

__device__ __forceinline__ RowP row_p(const RowSide& s, bool greedy) {
  RowP r;
  r.m = s.m, r.mz = s.mz, r.c = s.c, r.invT = s.invT, r.greedy = greedy;
  r.S = s.Z, r.Z = s.Z, r.invZ = s.invZ, r.vstar = s.vstar, r.Dstar = s.Dstar;
  r.kmax = 0u;
  return r;
}

// A warp reads a row from global memory in steps of kUnrollG groups per lane
// (lane l: groups x0, x0 + 256, ...), so several 16-byte loads are in flight;
// groups at or beyond V read as neutral values (never loaded).
constexpr int kUnrollG = 4;
template <int EB, bool PROBS>
__device__ __forceinline__ void load_groups_global(Grp<EB> (&g)[kUnrollG], const char* row, int x0,
                                                   int V) {
#pragma unroll
  for (int u = 0; u < kUnrollG; ++u) {
    const int x = x0 + u * 32 * kGroup;
    if (x < V) {
      lds_group<EB, PROBS>(g[u], row, 0, x, V);
    } else {
#pragma unroll
      for (int j = 0; j < EB * 2; ++j) g[u].w[j] = neutral_word<EB, PROBS>();
    }
  }
}

// ---------------------------------------------------------------------------
// Exact top-p boundary of one row read from global memory by one warp: a
// radix descent over the order key, 8 bits per level (2 levels for bf16, 4
// for fp32), each level summing the weights of the elements under the
// current key prefix per bin; the kept mass is then recomputed in a fixed
// order.  fh is 256 floats of the warp's shared scratch.  Sets Dstar, Z,
// invZ and vstar of r (r.kmax must hold vkey(m)).
// ---------------------------------------------------------------------------
template <int EB, bool PROBS>
__device__ __noinline__ void exact_top_p_warp(const char* row, int V, RowP& r, float R, float* fh) {
  const int lane = threadIdx.x & 31;
  constexpr int KB = EB == 2 ? 16 : 32;
  uint32_t prefix = 0u;
  float above = 0.0f;
  for (int shift = KB - 8; shift >= 0; shift -= 8) {
    for (int j = lane; j < kBins; j += 32) fh[j] = 0.0f;
    __syncwarp();
    const int hi = shift + 8;  // bits above this level's byte must equal the prefix's
#pragma unroll 1
    for (int x0 = lane * kGroup; x0 < V; x0 += kUnrollG * 32 * kGroup) {
      Grp<EB> g[kUnrollG];
      load_groups_global<EB, PROBS>(g, row, x0, V);
#pragma unroll
      for (int u = 0; u < kUnrollG; ++u) {
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const float v = gval<EB>(g[u], e);
          const uint32_t key = vkey<EB>(v);
          if (hi < KB && (key >> hi) != (prefix >> hi)) continue;
          const float w = weight<PROBS>(v, r);
          if (w > 0.0f) atomicAdd(&fh[(key >> shift) & 255u], w);
        }
      }
    }
    __syncwarp();
    // bins in descending key order: lane l holds bins 255 - 8l - q, q = 0..7
    float h[8], inc[8], t = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) h[q] = fh[255 - 8 * lane - q], t += h[q], inc[q] = t;
    float off = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, off, o);
      if (lane >= o) off += v;
    }
    off -= t;
    int first = 8;
#pragma unroll
    for (int q = 7; q >= 0; --q)
      if (above + off + inc[q] >= R) first = q;
    const uint32_t hit = __ballot_sync(0xffffffffu, first < 8);
    int src, q;
    if (hit) {
      src = __ffs(hit) - 1;
      q = __shfl_sync(0xffffffffu, first, src);
    } else {  // rounding left R unreachable: keep through the lowest non-empty bin
      int last = -1;
#pragma unroll
      for (int qq = 0; qq < 8; ++qq)
        if (h[qq] > 0.0f) last = qq;
      const uint32_t any = __ballot_sync(0xffffffffu, last >= 0);
      src = any ? 31 - __clz(any) : 0;
      q = any ? __shfl_sync(0xffffffffu, last, src) : 0;
    }
    float mine = off;  // mass of the bins above the chosen one (valid on lane src)
#pragma unroll
    for (int qq = 0; qq < 8; ++qq)
      if (qq < q) mine += h[qq];
    above += __shfl_sync(0xffffffffu, mine, src);
    prefix |= (255u - (uint32_t)(8 * src + q)) << shift;
    __syncwarp();  // fh is rewritten by the next level
  }
  float z = 0.0f;  // kept mass, per lane in a fixed order, then a fixed butterfly
#pragma unroll 1
  for (int x0 = lane * kGroup; x0 < V; x0 += kUnrollG * 32 * kGroup) {
    Grp<EB> g[kUnrollG];
    load_groups_global<EB, PROBS>(g, row, x0, V);
#pragma unroll
    for (int u = 0; u < kUnrollG; ++u) {
#pragma unroll
      for (int e = 0; e < kGroup; ++e) {
        const float v = gval<EB>(g[u], e);
        if (vkey<EB>(v) >= prefix) z += weight<PROBS>(v, r);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  r.Dstar = r.kmax - prefix;
  r.Z = z;
  r.invZ = 1.0f / z;
  r.vstar = vkey_value<EB>(prefix);
}

}  // namespace stream

using StreamFn = void (*)(stream::SParams);
StreamFn stream_bf16_bf16_logits();
StreamFn stream_bf16_f32_probs();
StreamFn stream_bf16_f32_logits();
StreamFn stream_f32_f32_logits();
StreamFn stream_f32_f32_probs();
StreamFn stream_f32_bf16_logits();

}  // namespace sv
