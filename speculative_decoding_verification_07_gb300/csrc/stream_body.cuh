#pragma once
// Streaming verification kernel: producer, consumers and finishers, the
// row-pair combine and the request resolution (see stream_kernel.cuh).
#include "stream_kernel.cuh"

namespace sv {
namespace stream {

// Barrier of consumer group g that also ORs a per-thread flag.
__device__ __forceinline__ bool gbar_or(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{.reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q;}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + g), "n"(kGT)
      : "memory");
  return r != 0u;
}

// ---------------------------------------------------------------------------
// Request state (finisher lane 0 writes, producers read)
// ---------------------------------------------------------------------------
constexpr unsigned long long kResolvedOne = 1ull << 32;  // CallSt::cnt, resolved count


// The first row of request b known to be decided and not accepted (kNA if none).
__device__ __forceinline__ int first_nonacc(const SParams& P, char* st, int b) {
  ReqSt* rq = req_st(st, b);
  if (P.kmax <= kFastK) {
    const uint32_t na = (uint32_t)(ld_relaxed64(&rq->w) >> 21) & 0x1FFFFFu;
    return na ? __ffs(na) - 1 : (int)kNA;
  }
  const uint32_t na = ld_relaxed(&rq->na);
  return na ? (int)(kNA - na) : (int)kNA;
}

// Rows of request b whose test saw q(y) == 0 (bit i: row i).
__device__ __forceinline__ unsigned long long qz_mask(const SParams& P, ReqSt* rq) {
  if (P.kmax <= kFastK) return (ld_relaxed64(&rq->w) >> 42) & 0x1FFFFFull;
  return ld_relaxed64(&rq->qz);
}

__device__ __forceinline__ uint32_t qz_bits(unsigned long long qz, int last_row) {
  const unsigned long long m = last_row >= 63 ? ~0ull : ((2ull << last_row) - 1ull);
  return (qz & m) ? SV_ST_Q_ZERO : 0u;
}

__device__ __forceinline__ void request_done(char* st) {
  __threadfence();
  atomicAdd(&call_st(st)->n_done, 1u);
}

// Resolve request b at its first non-accepted row f (rows 0 .. f-1 are
// accepted and row f is decided); sf is row f's state if the caller knows it.
static __device__ void resolve(const SParams& P, char* st, int b, int f, int sf) {
  CallSt* cs = call_st(st);
  ReqSt* rq = req_st(st, b);
  if (sf < 0) sf = (int)ld_relaxed(&pair_st(st, P, (size_t)b * (P.kmax + 1) + f)->state);
  if (sf == SV_ROW_REJECTED || sf == SV_ROW_BONUS) {
    // one atomic counts the resolution and claims the race's queue slot: a
    // waiter that sees every request resolved also sees every slot claimed
    const int seq = P.seq_len ? P.seq_len[b] : 0;
    const uint32_t rid = P.request_id ? P.request_id[b] : (uint32_t)b;
    const uint32_t q = (uint32_t)atomicAdd(&cs->cnt, kResolvedOne | 1ull);
    Slot* sl = slot_st(st, P.B, (int)q);
    const uint32_t kind = sf == SV_ROW_REJECTED ? kRaceResidual : kRaceBonus;
    st_relaxed64(&sl->w1, (unsigned long long)(uint32_t)(seq + 1 + f) | ((unsigned long long)rid << 32));
    st_release64(&sl->w0, kSlotFilled | ((unsigned long long)f << 32) | ((unsigned long long)b << 8) | kind);
    return;
  }
  if (sf == SV_ROW_TERMINAL) {
    const unsigned long long qz = qz_mask(P, rq);
    int32_t* ot = P.out_tokens + (size_t)b * (P.kmax + 1);
    for (int j = 0; j <= P.kmax; ++j) ot[j] = j <= f ? P.tokens[(size_t)b * P.kmax + j] : -1;
    const int eos = P.eos ? P.eos[b] : -1;
    const bool is_eos = eos >= 0 && P.tokens[(size_t)b * P.kmax + f] == eos;
    P.accepted[b] = f + 1;
    P.num_emitted[b] = f + 1;
    P.status[b] = qz_bits(qz, f) | (is_eos ? SV_ST_EOS : SV_ST_CAPPED);
  } else {  // invalid row
    bad_outputs(P, b, SV_ST_BAD_INPUT);
  }
  __threadfence();
  atomicAdd(&cs->cnt, kResolvedOne);
  request_done(st);
}

// The row at which decision word w resolves its request, or -1.
__device__ __forceinline__ int resolved_at(unsigned long long w) {
  const uint32_t na = (uint32_t)(w >> 21) & 0x1FFFFFu;
  if (!na) return -1;
  const int f = __ffs(na) - 1;
  const uint32_t need = (1u << f) - 1u;
  return ((uint32_t)w & need) == need ? f : -1;
}

// Publish row i's decision in request b's state; resolve the request if this
// completes "rows 0 .. f-1 accepted, row f decided".  The row's record and
// state were written before: the fence orders them before the decision.
static __device__ void publish(const SParams& P, char* st, int b, int i, int state, bool qzero) {
  ReqSt* rq = req_st(st, b);
  __threadfence();
  if (P.kmax <= kFastK) {
    unsigned long long bit = state == SV_ROW_ACCEPTED ? (1ull << i) : (1ull << (21 + i));
    if (qzero) bit |= 1ull << (42 + i);
    const unsigned long long old = atomicOr(&rq->w, bit);
    const int f = resolved_at(old | bit);
    if (f < 0 || resolved_at(old) >= 0) return;  // exactly one publisher sees the transition
    if (atomicCAS(&rq->resolved, 0u, 1u) != 0u) return;  // a timeout report came first
    __threadfence();
    resolve(P, st, b, f, f == i ? state : -1);
    return;
  }
  if (qzero) atomicOr(&rq->qz, 1ull << i);
  __threadfence();
  unsigned long long acc;
  uint32_t na;
  if (state == SV_ROW_ACCEPTED) {
    acc = atomicOr(&rq->acc, 1ull << i) | (1ull << i);
    fence_sc();
    na = ld_relaxed(&rq->na);
  } else {
    const uint32_t mine = kNA - (uint32_t)i;
    const uint32_t old = atomicMax(&rq->na, mine);
    fence_sc();
    acc = ld_relaxed64(&rq->acc);
    na = old > mine ? old : mine;
  }
  if (na == 0u) return;
  const int f = (int)(kNA - na);
  const unsigned long long need = f >= 64 ? ~0ull : ((1ull << f) - 1ull);
  if ((acc & need) == need && atomicCAS(&rq->resolved, 0u, 1u) == 0u) {
    __threadfence();
    resolve(P, st, b, f, f == i ? state : -1);
  }
}

// Queue a window band of row pair (b, i): the pair's band keys and flags are
// written before; the slot's ready flag releases them to the producers.
static __device__ void queue_window(const SParams& P, char* st, int b, int i, uint32_t win, uint32_t lo_t,
                                    uint32_t hi_t, uint32_t lo_d, uint32_t hi_d) {
  const uint32_t q = (uint32_t)atomicAdd(&call_st(st)->cnt, 1ull);
  Slot* sl = slot_st(st, P.B, (int)q);  // capacity: kMaxBands bands per row pair
  st_relaxed64(&sl->w1, (unsigned long long)(lo_t | (hi_t << 16)) | ((unsigned long long)(lo_d | (hi_d << 16)) << 32));
  st_release64(&sl->w0, kSlotFilled | ((unsigned long long)i << 32) | ((unsigned long long)b << 8) |
                            (win << 3) | kWindowSlot);
}

// ---------------------------------------------------------------------------
// Producer warp
// ---------------------------------------------------------------------------
constexpr uint32_t kNoTicket = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t take_ticket(const SParams& P) {
  uint32_t t = 0u;
  if ((threadIdx.x & 31) == 0) t = atomicAdd(&P.hdr->ticket, 1u);
  return __shfl_sync(0xffffffffu, t, 0);
}


// Is row (i, b) worth a ticket, given the request's k, cap and first known
// non-accepted row fna?  1: a row to load, 2: a bad request's report (i = 0),
// 0: nothing (absent, or behind a known rejection).
__device__ __forceinline__ int interest_of(const SParams& P, int i, int kb, int cap, int fna) {
  if (kb < 0 || kb > P.kmax || cap < 1) return i == 0 ? 2 : 0;
  const int last = cap <= kb ? cap - 1 : kb;
  if (i > last) return 0;
  if (!(P.flags & SV_FLAG_NO_SKIP) && fna < i) return 0;
  return 1;
}

__device__ __forceinline__ int row_interest(const SParams& P, char* st, int i, int b) {
  const int kb = P.k ? P.k[b] : P.kmax;
  const int cap = P.max_new ? P.max_new[b] : 0x7FFFFFFF;
  const int fna = (i > 0 && !(P.flags & SV_FLAG_NO_SKIP)) ? first_nonacc(P, st, b) : (int)kNA;
  return interest_of(P, i, kb, cap, fna);
}

// After an uninteresting row R = i * B + b: find the next interesting row
// (the warp checks 32 rows at a time), move the ticket counter up to it and
// own its first ticket if nobody passed it yet; else take a fresh ticket.
static __device__ uint32_t jump_ticket(const SParams& P, char* st, int R) {
  const int lane = threadIdx.x & 31;
  const int nrows = (P.kmax + 1) * P.B;
  int target = nrows;
  for (int base = R + 1; base < nrows; base += 32) {
    const int r = base + lane;
    const bool hit = r < nrows && row_interest(P, st, r / P.B, r % P.B) != 0;
    const uint32_t m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      target = base + __ffs(m) - 1;
      break;
    }
    if (base - R > 256) {  // long run of empty rows: jump this far and look again
      target = base + 32 < nrows ? base + 32 : nrows;
      break;
    }
  }
  const uint32_t tt = (uint32_t)target * (uint32_t)P.n_blk;
  uint32_t t = 0u;
  if (lane == 0) {
    const uint32_t old = atomicMax(&P.hdr->ticket, tt + 1u);
    t = old <= tt ? tt : atomicAdd(&P.hdr->ticket, 1u);
  }
  return __shfl_sync(0xffffffffu, t, 0);
}

// A waiter gave up on a queue slot: requests never resolved are reported as
// timed out (their outputs say so) and the call's error word is set.
static __device__ void timeout_sweep(const SParams& P, char* st) {
  const int lane = threadIdx.x & 31;
  for (int b = lane; b < P.B; b += 32) {
    ReqSt* rq = req_st(st, b);
    if (atomicCAS(&rq->resolved, 0u, 2u) == 0u) {
      bad_outputs(P, b, SV_ST_TIMEOUT);
      __threadfence();
      atomicAdd(&call_st(st)->cnt, kResolvedOne);
    }
  }
  if (lane == 0) report(P.err, SV_ERR_TIMEOUT);
}

// Fill h with the queued work of ticket (slot q, chunk block blk) from the
// slot's two words; returns the number of chunks.
template <int EBT, int EBD>
__device__ __forceinline__ int queued_item(const SParams& P, int blk, unsigned long long w0,
                                           unsigned long long w1, SHdr& h) {
  const int kind = (int)(w0 & 7u);
  h.b = (int)((w0 >> 8) & 0xFFFFFFu);
  h.i = (int)((w0 >> 32) & 0x7FFFFFFFu);
  h.c = blk * kBatch;
  if (kind == kWindowSlot) {
    h.kind = kWinItem;
    h.win = (int)((w0 >> 3) & 3u);
    h.has_d = (h.win & 2) ? 1 : 0;
    h.lo_t = (uint32_t)(w1 & 0xFFFFu), h.hi_t = (uint32_t)((w1 >> 16) & 0xFFFFu);
    h.lo_d = (uint32_t)((w1 >> 32) & 0xFFFFu), h.hi_d = (uint32_t)(w1 >> 48);
  } else {
    h.kind = kRaceItem;
    h.race = kind;
    h.has_d = kind == kRaceResidual;
    h.pos = (int)(uint32_t)w1;
    h.rid = (uint32_t)(w1 >> 32);
  }
  return min(kBatch, P.n_ch - h.c);
}

template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void producer(const SParams& P, SSmem& sm, char* dyn, char* st) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int NS = num_stages<EBT, EBD>();
  constexpr int SB = stage_bytes<EBT, EBD>();
  const int lane = threadIdx.x & 31;
  CallSt* cs = call_st(st);
  const uint32_t nb = (uint32_t)P.n_blk;
  uint32_t used = 0u, eph = 0u;  // per stage: used once / parity of its next empty phase
  int s = 0;
  // A ticket is a block of up to kBatch chunks of one row pair, settled in
  // one round trip and issued as consecutive items.  Two static tickets in
  // hand: the next one's atomic is in flight while the current one is
  // settled.  Queued work (window and race chunks) comes first: a queued
  // ticket is taken as soon as the queue shows work (its atomic completes
  // while the stages are issued), its slot is polled with the static
  // ticket's parameters in one round trip, and it is waited for only when
  // the static work has run out.
  uint32_t t = take_ticket(P), tn = take_ticket(P);
  uint32_t dh = kNoTicket, dh_raw = 0u;  // dh_raw: lane 0's queued-ticket atomic, in flight
  bool dh_pending = false;
  unsigned long long wait_t0 = 0ull;
  for (;;) {
    SHdr h;
    h.kind = kEnd;
    h.b = h.i = h.c = 0;
    h.x0 = h.n = h.has_d = h.kb = 0;
    h.T = 0.0f, h.top_p = 1.0f;
    h.race = 0, h.pos = 0, h.rid = 0u, h.y = 0;
    h.win = 0, h.lo_t = h.hi_t = h.lo_d = h.hi_d = 0u;
    bool from_static = false;
    int nitems = kNG;  // an end goes to every consumer group
    // ------------------------------------------------------------ settle
    for (int spins = 0;; ++spins) {
      if (dh_pending) {
        dh = __shfl_sync(0xffffffffu, dh_raw, 0);
        dh_pending = false;
      }
      if (tn < t) {
        const uint32_t x = t;
        t = tn, tn = x;
      }
      const bool static_left = t < P.n_static;
      const int R = static_left ? (int)(t / nb) : 0;
      const int blk = (int)(t - (uint32_t)R * nb);
      const int i = R / P.B, b = R - i * P.B;
      const uint32_t q = dh != kNoTicket ? dh / nb : 0u;
      // one round trip: the static row's parameters (lanes 0-5), the held
      // slot (6, 7), the queue counters (8, 9)
      int iv = 0;
      float fv = 0.0f;
      unsigned long long wv = 0ull;
      if (static_left) {
        if (lane == 0) iv = P.k ? P.k[b] : P.kmax;
        if (lane == 1) iv = P.max_new ? P.max_new[b] : 0x7FFFFFFF;
        if (lane == 2) iv = (i > 0 && !(P.flags & SV_FLAG_NO_SKIP)) ? first_nonacc(P, st, b) : (int)kNA;
        if (lane == 3) fv = P.temperature[b];
        if (lane == 4) fv = P.top_p ? P.top_p[b] : 1.0f;
        if (lane == 5 && i < P.kmax) iv = P.tokens[(size_t)b * P.kmax + i];
      }
      if (dh != kNoTicket && q < P.n_slots) {
        if (lane == 6) wv = ld_acquire64(&slot_st(st, P.B, (int)q)->w0);
        if (lane == 7) wv = ld_relaxed64(&slot_st(st, P.B, (int)q)->w1);
      }
      if (lane == 8) wv = ld_relaxed64(&cs->cnt);
      if (lane == 9) wv = ld_relaxed(&P.hdr->dticket);
      const unsigned long long w0 = __shfl_sync(0xffffffffu, wv, 6);
      const unsigned long long w1 = __shfl_sync(0xffffffffu, wv, 7);
      const unsigned long long cnt = __shfl_sync(0xffffffffu, wv, 8);
      const uint32_t dnext = (uint32_t)__shfl_sync(0xffffffffu, wv, 9);
      const uint32_t claimed = (uint32_t)cnt;
      if (dh != kNoTicket) {
        if ((w0 & kSlotFilled) && w1 != 0ull) {
          nitems = queued_item<EBT, EBD>(P, (int)(dh - q * nb), w0, w1, h);
          dh = kNoTicket;
          if (dnext < claimed * nb) {  // more queued work: take the next ticket now
            if (lane == 0) dh_raw = atomicAdd(&P.hdr->dticket, 1u);
            dh_pending = true;
          }
          break;
        }
        if (!static_left) {  // nothing else to do: wait for the slot, or end
          if ((uint32_t)(cnt >> 32) >= (uint32_t)P.B && claimed <= q) break;  // END: no slot will come
          if (wait_t0 == 0ull) wait_t0 = gtimer();
          if (__shfl_sync(0xffffffffu, gtimer() - wait_t0 > P.slot_wait_ns ? 1 : 0, 0)) {
            timeout_sweep(P, st);
            break;  // END
          }
          __nanosleep(spins < 64 ? 64 : 256);
          continue;
        }
      } else if (!static_left || dnext < claimed * nb) {
        if (lane == 0) dh_raw = atomicAdd(&P.hdr->dticket, 1u);
        dh_pending = true;
        if (!static_left) continue;
      }
      // ---------------------------------------------------- static work
      const int kb = __shfl_sync(0xffffffffu, iv, 0);
      const int cap = __shfl_sync(0xffffffffu, iv, 1);
      const int fna = __shfl_sync(0xffffffffu, iv, 2);
      const float T = __shfl_sync(0xffffffffu, fv, 3);
      const float tp = __shfl_sync(0xffffffffu, fv, 4);
      const int y = __shfl_sync(0xffffffffu, iv, 5);
      const int what = interest_of(P, i, kb, cap, fna);
      if (what == 1 || (what == 2 && blk == 0)) {
        h.kind = what == 1 ? kRowItem : kBadItem;
        h.b = b, h.i = i, h.c = blk * kBatch;
        nitems = 1;
        if (what == 1) {
          nitems = min(kBatch, P.n_ch - h.c);
          h.kb = kb;
          h.has_d = i < kb;
          h.T = T;
          h.top_p = tp;
          h.y = h.has_d ? y : 0;
        }
        from_static = true;
        break;
      }
      t = jump_ticket(P, st, R);
      if (lane == 0) SV_TR(3, R, t);
    }
    wait_t0 = 0ull;
    if (lane == 0) SV_TR(1, (h.kind << 20) | (h.i << 12) | h.c, h.b);
    const int c0 = h.c;
    for (int rep = 0; rep < nitems; ++rep) {
      if (rep > 0) s = s + 1 == NS ? 0 : s + 1;
      if (h.kind != kEnd) {
        h.c = c0 + rep;
        h.x0 = h.c * CH;
        h.n = min(CH, P.V - h.x0);
      }
      // ------------------------------------------------ wait for the stage
      if (used & (1u << s)) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_ns(&sm.empty[s], (eph >> s) & 1u, P.err, kStageWaitNs, 256u);
        if (lane == 0) SV_TR(4, s, 0);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        eph ^= 1u << s;
        if (!ok) h.kind = kEnd;  // the consumers stopped: end this CTA
      }
      used |= 1u << s;
      if (h.kind == kRaceItem) {  // the decided row's record, 16 words over 16 lanes
        const uint32_t* src = reinterpret_cast<const uint32_t*>(P.rows + (size_t)h.b * (P.kmax + 1) + h.i);
        if (lane < 16) reinterpret_cast<uint32_t*>(&sm.hdr[s].rr)[lane] = __ldcg(src + lane);
      }
      if (lane == 0) {
        SHdr& d = sm.hdr[s];
        d.kind = h.kind, d.b = h.b, d.i = h.i, d.c = h.c;
        d.x0 = h.x0, d.n = h.n, d.has_d = h.has_d, d.kb = h.kb;
        d.T = h.T, d.top_p = h.top_p, d.race = h.race, d.pos = h.pos, d.rid = h.rid, d.y = h.y;
        d.win = h.win, d.lo_t = h.lo_t, d.hi_t = h.hi_t, d.lo_d = h.lo_d, d.hi_d = h.hi_d;
      }
      __syncwarp();
      if (lane == 0) {
        if (h.kind == kRowItem || h.kind == kRaceItem || h.kind == kWinItem) {
          // window items load only the sides their band counts
          const bool lt = h.kind != kWinItem || (h.win & 1);
          char* sT = dyn + (size_t)s * SB;
          char* sD = sT + (size_t)CH * EBT;
          const uint32_t bt = lt ? (uint32_t)((h.n * EBT + 15) & ~15) : 0u;
          const uint32_t bd = h.has_d ? (uint32_t)((h.n * EBD + 15) & ~15) : 0u;
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_expect_tx(&sm.full[s], bt + bd);
          if (lt) {
            const char* trow = P.target + ((size_t)h.b * (P.kmax + 1) + h.i) * (size_t)P.t_ld * EBT;
            bulk_g2s(sT, trow + (size_t)h.x0 * EBT, bt, &sm.full[s]);
          }
          if (h.has_d) {
            const char* drow = P.draft + ((size_t)h.b * P.kmax + h.i) * (size_t)P.d_ld * EBD;
            bulk_g2s(sD, drow + (size_t)h.x0 * EBD, bd, &sm.full[s]);
          }
        } else {
          mbar_arrive1(&sm.full[s]);
        }
      }
      if (lane == 0) SV_TR(2, s, t);
    }
    if (h.kind == kEnd) break;
    s = s + 1 == NS ? 0 : s + 1;
    if (from_static) t = tn, tn = take_ticket(P);
  }
}

// ---------------------------------------------------------------------------
// Consumers
// ---------------------------------------------------------------------------
// Packed bf16x2 maximum of the four words of a group (each half: the
// maximum of the group's even or odd elements).
__device__ __forceinline__ uint32_t group_max2(const Grp<2>& g) {
  return bmax2(bmax2(g.w[0], g.w[1]), bmax2(g.w[2], g.w[3]));
}

// Element e (0..7) of a bf16 group held in registers, as its 16 bits.
__device__ __forceinline__ uint32_t group_half(const uint4& g, int e) {
  const uint32_t w = (e & 4) ? ((e & 2) ? g.w : g.z) : ((e & 2) ? g.y : g.x);
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// First pass over one chunk of a row pair: the stage is read once and the
// thread's groups of both rows stay in registers for the maxima and the
// weight sums, which are taken relative to the warp's own maxima (the
// finisher rescales the warp partials to the chunk maxima).  No barrier.
template <int EBT, int EBD, bool PROBS>
__device__ void process_row(const SParams& P, SSmem& sm, const SHdr& h, int s, int f, const char* sT,
                            const char* sD, int g) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int GPT = CH / kGroup / kGT;
  const int ctid = (int)threadIdx.x & (kGT - 1), lane = ctid & 31, warp = (int)threadIdx.x >> 5;
  const int gw = warp & (kGW - 1);
  const bool has_d = h.has_d;
  const float T = h.T;
  const bool greedy = T == 0.0f;
  const float ct = greedy ? 0.0f : kLog2e / T;
  const float invT = greedy ? 0.0f : 1.0f / T;
  const float cd = PROBS ? 1.0f : ct;
  SliceIter it;
  it.x0 = h.x0, it.x1 = h.x0 + h.n, it.nblk = GPT, it.V = P.V;
  it.stride = kGT * kGroup, it.tid = ctid;
  Fin& F = sm.fin[f];

  Grp<EBT> gt[GPT];
  Grp<EBD> gd[GPT];
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    lds_group_or_neutral<EBT, false>(gt[j], sT, it.x0, it.x(j), it.x1);
    if (has_d) lds_group_or_neutral<EBD, PROBS>(gd[j], sD, it.x0, it.x(j), it.x1);
  }
  uint32_t mt2 = 0xFF80FF80u, md2 = PROBS ? 0u : 0xFF80FF80u;
  float rmt = -INFINITY, rmd = PROBS ? 0.0f : -INFINITY;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    max_group<EBT>(gt[j], mt2, rmt);
    if (has_d) max_group<EBD>(gd[j], md2, rmd);
  }
  float mt = max_value<EBT>(mt2, rmt), md = max_value<EBD>(md2, rmd);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, o));
  }
  if (ctid == 0) SV_TR(11, 0, g);
  const float mzd = weight_max<PROBS>(md, greedy, invT);
  float sumt = 0.0f, sumd = 0.0f;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    sumt += sum_group<EBT, false>(gt[j], greedy, mt, ct, invT);
    if (has_d) sumd += sum_group<EBD, PROBS>(gd[j], greedy, mzd, cd, invT);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    sumt += __shfl_xor_sync(0xffffffffu, sumt, o);
    sumd += __shfl_xor_sync(0xffffffffu, sumd, o);
  }
  if (lane == 0) F.wp[gw] = make_float4(mt, sumt, md, sumd);
  if (ctid == 0) {  // the accept-test operands, when the proposal lies in this chunk
    const bool hy = has_d && h.y >= it.x0 && h.y < it.x1;
    float vt = 0.0f, vd = 0.0f;
    if (hy) {
      const int e = h.y - it.x0;
      vt = EBT == 2 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(sT)[e] << 16)
                    : reinterpret_cast<const float*>(sT)[e];
      vd = EBD == 2 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(sD)[e] << 16)
                    : reinterpret_cast<const float*>(sD)[e];
    }
    F.vt = vt, F.vd = vd, F.has_y = hy ? 1 : 0;
    F.kind = kRowItem, F.b = h.b, F.i = h.i, F.c = h.c;
    F.has_d = h.has_d, F.kb = h.kb, F.T = T, F.top_p = h.top_p, F.y = h.y;
  }
  release_stage(sm, s);
  __syncwarp();
  if (lane == 0) mbar_arrive1(&sm.fin_full[f]);
  if (ctid == 0) SV_TR(13, f, g);
}

// Window counts of the candidate groups a warp collected: entry v names a
// group by its offset in the chunk (bits 0-14) and its row (bit 15: draft).
// Each lane takes whole groups, re-reads them from the stage and counts the
// elements of the band [lo, hi] into bins j = hi - key.
__device__ __forceinline__ void band_groups(const uint16_t* buf, int total, const char* sT, const char* sD,
                                            uint32_t thr_t, uint32_t thr_d, uint32_t hi_t, uint32_t hi_d,
                                            int x0, int x1, uint32_t* hist_t, uint32_t* hist_d) {
  for (int e = threadIdx.x & 31; e < total; e += 32) {
    const uint32_t v = buf[e];
    const bool dr = (v >> 15) != 0u;
    const int off = (int)(v & 0x7FFFu);
    const uint4 g = *reinterpret_cast<const uint4*>((dr ? sD : sT) + (size_t)off * 2);
    uint32_t m = window_bits_bf16(g, dr ? thr_d : thr_t, x0 + off, x1);
    const uint32_t hi = dr ? hi_d : hi_t;
    uint32_t* hist = dr ? hist_d : hist_t;
    while (m) {
      const int k = __ffs(m) - 1;
      m &= m - 1u;
      const uint32_t j = hi - bf16_order_key(group_half(g, k));
      if (j < (uint32_t)kBins) atomicAdd(&hist[j], 1u);
    }
  }
}

// A window item: the counts of one chunk's bf16 values in the row pair's
// band [lo, hi] (for the sides the band counts).  Groups whose maximum is
// below the band are skipped; the rest go through the warp's buffer.
template <int EBT, int EBD, bool PROBS>
__device__ void process_win(const SParams& P, SSmem& sm, const SHdr& h, int s, int f, const char* sT,
                            const char* sD, int g) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int GPT = CH / kGroup / kGT;
  static_assert(2 * GPT * 32 <= 256, "candidate groups fit the warp buffer");
  const int ctid = (int)threadIdx.x & (kGT - 1), lane = ctid & 31, warp = (int)threadIdx.x >> 5;
  Fin& F = sm.fin[f];
  if constexpr (EBT == 2 && EBD == 2 && !PROBS) {
    SliceIter it;
    it.x0 = h.x0, it.x1 = h.x0 + h.n, it.nblk = GPT, it.V = P.V;
    it.stride = kGT * kGroup, it.tid = ctid;
    const bool wt = h.win & 1, wd = h.win & 2;
    const uint32_t tb = __float_as_uint(vkey_value<2>(h.lo_t)) >> 16;
    const uint32_t db = __float_as_uint(vkey_value<2>(h.lo_d)) >> 16;
    const uint32_t thr_t = tb | (tb << 16), thr_d = db | (db << 16);
    uint32_t cm = 0u;  // bit j: target group j may hold band elements; bit GPT + j: draft
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
      Grp<2> q;
      if (wt) {
        lds_group_or_neutral<2, false>(q, sT, it.x0, it.x(j), it.x1);
        cm |= (bge2(group_max2(q), thr_t) != 0u ? 1u : 0u) << j;
      }
      if (wd) {
        lds_group_or_neutral<2, false>(q, sD, it.x0, it.x(j), it.x1);
        cm |= (bge2(group_max2(q), thr_d) != 0u ? 1u : 0u) << (GPT + j);
      }
    }
    const int n = __popc(cm);
    const int incl = warp_incl_scan(n);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total) {
      uint16_t* buf = sm.wb[warp];
      int pos = incl - n;
      while (cm) {
        const int bit = __ffs(cm) - 1;
        cm &= cm - 1u;
        buf[pos++] = (uint16_t)(((bit >= GPT) ? 0x8000 : 0) | (it.x(bit % GPT) - it.x0));
      }
      __syncwarp();
      band_groups(buf, total, sT, sD, thr_t, thr_d, h.hi_t, h.hi_d, it.x0, it.x1, F.hist[0], F.hist[1]);
    }
    if (ctid == 0) SV_TR(15, total, g);
  }
  if (ctid == 0) {
    F.kind = kWinItem, F.b = h.b, F.i = h.i, F.c = h.c;
    F.win = h.win;
  }
  release_stage(sm, s);
  __syncwarp();
  if (lane == 0) mbar_arrive1(&sm.fin_full[f]);
  if (ctid == 0) SV_TR(16, f, g);
}

template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void process_race(const SParams& P, SSmem& sm, const SHdr& h, int s, int f, const char* sT,
                                          const char* sD, int g) {
  constexpr int GPT = chunk_elems<EBT, EBD>() / kGroup / kGT;
  const int ctid = (int)threadIdx.x & (kGT - 1), lane = ctid & 31, warp = (int)threadIdx.x >> 5;
  const RowRec rr = h.rr;
  const int hb = h.b, hi = h.i, hc = h.c, hrace = h.race, hpos = h.pos;
  const uint32_t hrid = h.rid;
  const bool greedy = rr.t.invT == 0.0f;
  RowP rt = row_p(rr.t, greedy), rd = row_p(rr.d, greedy);
  rt.kmax = vkey<EBT>(rt.m);
  rd.kmax = vkey<EBD>(rd.m);
  const bool residual = h.race == kRaceResidual;
  SliceIter it;
  it.x0 = h.x0, it.x1 = h.x0 + h.n, it.nblk = GPT, it.V = P.V;
  it.stride = kGT * kGroup, it.tid = ctid;
  RacePart best = {0.0f, 1.0f, 0x7FFFFFFF};
  race_slice<EBT, EBD, PROBS>(sT, sD, it, residual, rt, rd, (uint32_t)h.pos, h.rid, P.seed_lo, P.seed_hi,
                              sm.wb[warp], best);
  release_stage(sm, s);
  warp_race(best.w, best.E, best.idx);
  if (lane == 0) sm.rp[warp] = best;
  gbar(g);
  if (ctid == 0) {
    const RacePart* rp = sm.rp + g * kGW;
    RacePart o = rp[0];
    for (int w = 1; w < kGW; ++w)
      if (better(rp[w].w, rp[w].E, rp[w].idx, o.w, o.E, o.idx)) o = rp[w];
    Fin& F = sm.fin[f];
    F.kind = kRaceItem, F.b = hb, F.i = hi, F.c = hc;
    F.race = hrace, F.pos = hpos, F.rid = hrid;
    F.rw = o.w, F.rE = o.E, F.ridx = o.idx;
    F.rr = rr;
    mbar_arrive_n(&sm.fin_full[f], kGW);
  }
}

template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void consumer(const SParams& P, SSmem& sm, char* dyn) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int NS = num_stages<EBT, EBD>();
  constexpr int SB = stage_bytes<EBT, EBD>();
  // Group g works items n = g, g + kNG, ...: stage n % NS, hand-off slot n % kNF.
  const int g = ((int)threadIdx.x >> 5) / kGW;
  const bool leader = ((int)threadIdx.x & (kGT - 1)) == 0;
  uint32_t fph = 0u, fused = 0u, feph = 0u;
  int s = g, f = g;
  for (;;) {
    // The group's first thread waits for the stage's data and for a free
    // hand-off slot; the group's other warps wait in the barrier (issuing
    // nothing), which also carries the outcome, so every thread of the group
    // takes the same path (a wait that did not complete in time ends this
    // CTA's work).  The barrier orders the stage's contents, seen complete
    // by the first thread, before every thread's reads.
    bool ok = true;
    if (leader) {
      ok = mbar_wait_ns(&sm.full[s], (fph >> s) & 1u, P.err, kStageWaitNs, 64u);
      SV_TR(17, s, g);
      if (fused & (1u << f))
        ok = mbar_wait_ns(&sm.fin_empty[f], (feph >> f) & 1u, P.err, kStageWaitNs, 64u) && ok;
    }
    fph ^= 1u << s;
    if (fused & (1u << f)) feph ^= 1u << f;
    fused |= 1u << f;
    const bool bad = gbar_or(g, !ok);
    // the stage's header stays in shared memory (read in place: a local copy
    // would live in local memory); its fields are read before the stage is
    // handed back, after which the producer may rewrite it
    const SHdr& h = sm.hdr[s];
    if (leader) SV_TR(10, h.kind | (g << 8), (h.b << 8) | (h.i << 4) | h.c);
    if (bad || h.kind == kEnd) {
      // tell the finishers to stop: the group's next kFW slots go to
      // kFW different finishers, each of which stops at the first end it meets
      if (leader) {
        for (int w = 0; w < kFW; ++w) {
          if (w > 0) {
            f = f + kNG >= kNF ? f + kNG - kNF : f + kNG;
            if (fused & (1u << f)) {
              (void)mbar_wait_ns(&sm.fin_empty[f], (feph >> f) & 1u, P.err, kStageWaitNs);
              feph ^= 1u << f;
            }
            fused |= 1u << f;
          }
          sm.fin[f].kind = kEnd;
          mbar_arrive_n(&sm.fin_full[f], kGW);
        }
      }
      break;
    }
    const char* sT = dyn + (size_t)s * SB;
    const char* sD = sT + (size_t)CH * EBT;
    if (h.kind == kRowItem) {
      process_row<EBT, EBD, PROBS>(P, sm, h, s, f, sT, sD, g);
    } else if (h.kind == kWinItem) {
      process_win<EBT, EBD, PROBS>(P, sm, h, s, f, sT, sD, g);
    } else if (h.kind == kRaceItem) {
      process_race<EBT, EBD, PROBS>(P, sm, h, s, f, sT, sD, g);
    } else {  // a bad request's report
      if (leader) {
        Fin& F = sm.fin[f];
        F.kind = kBadItem, F.b = h.b;
      }
      release_stage(sm, s);
      if (leader) mbar_arrive_n(&sm.fin_full[f], kGW);
    }
    s = s + kNG >= NS ? s + kNG - NS : s + kNG;
    f = f + kNG >= kNF ? f + kNG - kNF : f + kNG;
  }
}

// ---------------------------------------------------------------------------
// Finishers
// ---------------------------------------------------------------------------
// Warp race over a whole row in global memory, from p (the correction when the
// residual is numerically empty).  Rare: plain per-element Philox.
template <int EBT>
__device__ __noinline__ int race_row_warp(const char* trow, int V, const RowP& rt, uint32_t pos,
                                          uint32_t rid, uint32_t k0, uint32_t k1) {
  const int lane = threadIdx.x & 31;
  float bw = 0.0f, bE = 1.0f;
  int bidx = 0x7FFFFFFF;
#pragma unroll 1
  for (int x = lane * kGroup; x < V; x += 32 * kGroup) {
    Grp<EBT> g;
    lds_group<EBT, false>(g, trow, 0, x, V);
#pragma unroll 1
    for (int e = 0; e < kGroup; ++e) {
      const float v = gval<EBT>(g, e);
      const float w = kept<EBT>(v, rt) ? weight<false>(v, rt) : 0.0f;
      if (!(w > 0.0f)) continue;
      const int xi = x + e;
      const uint4 r = philox4x32_10(make_uint4((uint32_t)xi >> 2, pos, rid, 0u), k0, k1);
      const uint32_t sel = (xi & 3) == 0 ? r.x : (xi & 3) == 1 ? r.y : (xi & 3) == 2 ? r.z : r.w;
      const float E = -logf(uniform_from_bits(sel));
      if (better(w, E, xi, bw, bE, bidx)) bw = w, bE = E, bidx = xi;
    }
  }
  warp_race(bw, bE, bidx);
  return bidx;
}

// The request's scalars a decision needs (one load per lane, then shared).
struct ReqScalars {
  int seq, rid, eos, cap;
};
__device__ __forceinline__ ReqScalars req_scalars(const SParams& P, int b) {
  const int lane = threadIdx.x & 31;
  int rv = 0;
  if (lane == 0) rv = P.seq_len ? P.seq_len[b] : 0;
  if (lane == 1) rv = P.request_id ? (int)P.request_id[b] : b;
  if (lane == 2) rv = P.eos ? P.eos[b] : -1;
  if (lane == 3) rv = P.max_new ? P.max_new[b] : 0x7FFFFFFF;
  ReqScalars r;
  r.seq = __shfl_sync(0xffffffffu, rv, 0), r.rid = __shfl_sync(0xffffffffu, rv, 1);
  r.eos = __shfl_sync(0xffffffffu, rv, 2), r.cap = __shfl_sync(0xffffffffu, rv, 3);
  return r;
}

// Row params of both sides from the merged first pass (no top-p filter yet).
template <int EBT, int EBD, bool PROBS>
__device__ __forceinline__ void row_params(float Mt, float St, float Md, float Sd, bool has_d, float T,
                                           RowP& rt, RowP& rd) {
  const bool greedy = T == 0.0f;
  const float ct = greedy ? 0.0f : kLog2e / T;
  const float invT = greedy ? 0.0f : 1.0f / T;
  rt.greedy = rd.greedy = greedy;
  rt.m = rt.mz = Mt, rt.S = St;
  if (has_d) {
    rd.m = Md, rd.mz = weight_max<PROBS>(Md, greedy, invT), rd.S = Sd;
  } else {
    rd.m = rd.mz = PROBS ? 0.0f : -INFINITY, rd.S = 1.0f;
  }
  rt.c = ct, rt.invT = invT, rt.kmax = vkey<EBT>(rt.m), rt.Dstar = kNoFilter, rt.vstar = -INFINITY;
  rt.Z = rt.S, rt.invZ = 1.0f / rt.S;
  rd.c = PROBS ? 1.0f : ct, rd.invT = invT, rd.kmax = vkey<EBD>(rd.m), rd.Dstar = kNoFilter;
  rd.vstar = PROBS ? 0.0f : -INFINITY;
  rd.Z = rd.S, rd.invZ = 1.0f / rd.S;
}

// The accept test of row i (lane 0), its record, and the decision published.
template <int EBT, int EBD, bool PROBS>
__device__ void decide_row(const SParams& P, char* st, int b, int i, int kb, int y, bool has_d, bool row_bad,
                           const RowP& rt, const RowP& rd, float vt, float vd, const ReqScalars& rs) {
  const int lane = threadIdx.x & 31;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  if (lane == 0) {
    int state;
    bool qzero = false;
    float p_y = 0.0f, q_y = 0.0f, u = 0.0f;
    if (row_bad) {
      state = SV_ROW_INVALID;
    } else if (has_d) {
      p_y = prob<EBT, false>(vt, rt);
      q_y = prob<EBD, PROBS>(vd, rd);
      const int pos = rs.seq + 1 + i;
      u = uniform_from_bits(
          philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)rs.rid, 1u), P.seed_lo, P.seed_hi).x);
      qzero = q_y == 0.0f;
      state = (u * q_y < p_y) ? SV_ROW_ACCEPTED : SV_ROW_REJECTED;
      if (state == SV_ROW_ACCEPTED) {
        if ((rs.eos >= 0 && y == rs.eos) || (rs.cap <= kb && i == rs.cap - 1)) state = SV_ROW_TERMINAL;
      }
    } else {
      state = SV_ROW_BONUS;
    }
    RowRec rec;
    rec.t = RowSide{rt.m, rt.mz, rt.c, rt.invT, rt.Z, rt.invZ, rt.vstar, rt.Dstar};
    rec.d = RowSide{rd.m, rd.mz, rd.c, rd.invT, rd.Z, rd.invZ, rd.vstar, rd.Dstar};
    P.rows[pair] = rec;
    if (P.debug) {
      sv_row_debug d;
      d.p_y = p_y, d.q_y = q_y, d.u = u;
      d.p_kept = rt.greedy || rt.Dstar == kNoFilter ? 1.0f : rt.Z / rt.S;
      d.q_kept = !has_d || rd.greedy || rd.Dstar == kNoFilter ? 1.0f : rd.Z / rd.S;
      d.state = state;
      d.p_thr_key = rt.Dstar == kNoFilter ? -1 : (int32_t)(rt.kmax - rt.Dstar);
      d.q_thr_key = (!has_d || rd.Dstar == kNoFilter) ? -1 : (int32_t)(rd.kmax - rd.Dstar);
      P.debug[pair] = d;
    }
    st_relaxed(&pair_st(st, P, pair)->state, (uint32_t)state);
    SV_TR(33, state, pair);
    const bool withhold = (P.flags & SV_FLAG_TEST_WITHHOLD) && pair == 0;
    if (!withhold) publish(P, st, b, i, state, qzero);
  }
  __syncwarp();
}

// Lowest key of the first band of a row side: `depth` log2 units (plus a
// margin) below the row maximum's key hi, at most 255 keys below it.
__device__ __forceinline__ uint32_t band_lo(uint32_t hi, float depth, float c) {
  const uint32_t lo255 = hi >= 255u ? hi - 255u : 0u;
  if (!(depth > 0.0f) || !(c > 0.0f)) return lo255;
  const float fv = vkey_value<2>(hi) - (depth + kDepthMargin) / c;
  uint32_t k = 0u;
  if (fv > -INFINITY) k = key16(__uint_as_float(bf16_pair_of(fv) << 16));
  if (k < lo255) k = lo255;
  if (k > hi) k = hi;
  return k;
}

// The row pair's first pass is complete (all chunks arrived): merge the chunk
// partials.  Without top-p the row is decided at once; else its first window
// band is set up and queued.
template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void merge_pass1(const SParams& P, int b, int i, int has_d, int kb, float T,
                                         float top_p, int y, char* st) {
  const int lane = threadIdx.x & 31;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  const char* parts = P.parts + pair * P.n_ch * (size_t)P.part_bytes;
  const bool greedy = T == 0.0f;
  const bool pok = row_params_ok(T, top_p);
  const float ct = greedy ? 0.0f : kLog2e / T;
  const float invT = greedy ? 0.0f : 1.0f / T;
  const float cd = PROBS ? 1.0f : ct;
  // chunk c's partial on lane c
  float4 a = make_float4(-INFINITY, 0.0f, PROBS ? 0.0f : -INFINITY, 0.0f);
  float4 hv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (lane < P.n_ch) {
    const float4* p = reinterpret_cast<const float4*>(parts + (size_t)lane * P.part_bytes);
    a = __ldcg(p);
    hv = __ldcg(p + 1);
    if (!has_d) a.z = PROBS ? 0.0f : -INFINITY, a.w = 0.0f;
  }
  const ReqScalars rs = req_scalars(P, b);
  float Mt = a.x, Md = a.z;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, o));
    Md = fmaxf(Md, __shfl_xor_sync(0xffffffffu, Md, o));
  }
  float St = rescale(a.x, a.y, Mt, ct, greedy);
  float Sd = rescale(weight_max<PROBS>(a.z, greedy, invT), a.w, weight_max<PROBS>(Md, greedy, invT), cd, greedy);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    St += __shfl_xor_sync(0xffffffffu, St, o);
    Sd += __shfl_xor_sync(0xffffffffu, Sd, o);
  }
  RowP rt, rd;
  row_params<EBT, EBD, PROBS>(Mt, St, Md, Sd, has_d, T, rt, rd);
  if (lane == 0) SV_TR(30, 0, pair);
  // the accept-test operands from the chunk that holds the proposal
  const uint32_t ym = __ballot_sync(0xffffffffu, lane < P.n_ch && hv.z != 0.0f);
  const int ysrc = ym ? __ffs(ym) - 1 : 0;
  const float vt = __shfl_sync(0xffffffffu, hv.x, ysrc), vd = __shfl_sync(0xffffffffu, hv.y, ysrc);
  const bool y_ok = !has_d || (y >= 0 && y < P.V && ym != 0u);
  const bool bad_t = !(rt.S >= 1.0f && rt.S <= FLT_MAX) || !(rt.m <= FLT_MAX) || rt.m == -INFINITY;
  const bool bad_d = has_d && (!(rd.S >= 1.0f && rd.S <= FLT_MAX) || !(rd.m <= FLT_MAX) ||
                               (PROBS ? !(rd.m > 0.0f) : rd.m == -INFINITY));
  const bool row_bad = bad_t || bad_d || !pok || !y_ok;
  const bool window = !row_bad && !greedy && top_p < 1.0f && P.hist;
  if (!window) {
    decide_row<EBT, EBD, PROBS>(P, st, b, i, kb, y, has_d, row_bad, rt, rd, vt, vd, rs);
    return;
  }
  if constexpr (EBT == 2) {
    // first band: from each maximum down to the deepest nucleus of the call
    // so far (plus a margin), at most 255 keys
    // (not for a row behind a known rejection: it will never be needed)
    if (lane == 0 && ((P.flags & SV_FLAG_NO_SKIP) || i == 0 || first_nonacc(P, st, b) >= i)) {
      CallSt* cs = call_st(st);
      PairStats* ps = P.pstats + pair;
      ps->Mt = Mt, ps->St = St, ps->Md = Md, ps->Sd = Sd;
      ps->vt = vt, ps->vd = vd, ps->above_t = 0.0f, ps->above_d = 0.0f;
      PairSt* pr = pair_st(st, P, pair);
      const uint32_t hi_t = key16(Mt);
      pr->hi_t = hi_t;
      // nucleus depths: the deepest of this call so far and of the previous call
      const float dt = fmaxf(__uint_as_float(ld_relaxed(&cs->depth_t)), __uint_as_float(ld_relaxed(&P.hdr->depth_t)));
      const float dd = fmaxf(__uint_as_float(ld_relaxed(&cs->depth_d)), __uint_as_float(ld_relaxed(&P.hdr->depth_d)));
      pr->lo_t = band_lo(hi_t, dt, ct);
      if (has_d) {
        const uint32_t hi_d = key16(Md);
        pr->hi_d = hi_d;
        pr->lo_d = band_lo(hi_d, dd, cd);
      }
      pr->wside = has_d ? 3u : 1u;
      __threadfence();
      queue_window(P, st, b, i, pr->wside, pr->lo_t, hi_t, has_d ? pr->lo_d : 0u, has_d ? pr->hi_d : 0u);
    }
    __syncwarp();
  }
}

// Sum the window counts of one side over the chunks (lane l: bins 8l .. 8l+7)
// and scan the band for the top-p boundary: bin j holds key hi - j.  Returns
// the bin of the boundary (the kept mass through it in Z), or -1 with the
// band's whole mass in Z when the boundary lies below the band.
__device__ __forceinline__ int band_scan(const SParams& P, const char* parts, int side, uint32_t hi,
                                         const RowP& r, float R, float above, float* fh, float& Z) {
  const int lane = threadIdx.x & 31;
  uint32_t cnt[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) cnt[q] = 0u;
  const char* base = parts + kPartHead + side * 512 + 16 * lane;
  for (int c0 = 0; c0 < P.n_ch; c0 += 8) {
    uint4 v[8];  // the loads of 8 chunks together (one round trip)
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = c0 + u < P.n_ch ? __ldcg(reinterpret_cast<const uint4*>(base + (size_t)(c0 + u) * P.part_bytes))
                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      cnt[0] += v[u].x & 0xFFFFu, cnt[1] += v[u].x >> 16;
      cnt[2] += v[u].y & 0xFFFFu, cnt[3] += v[u].y >> 16;
      cnt[4] += v[u].z & 0xFFFFu, cnt[5] += v[u].z >> 16;
      cnt[6] += v[u].w & 0xFFFFu, cnt[7] += v[u].w >> 16;
    }
  }
  float h[8], inc[8], t = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t j = (uint32_t)(8 * lane + q);
    h[q] = (cnt[q] && j <= hi) ? (float)cnt[q] * weight<false>(vkey_value<2>(hi - j), r) : 0.0f;
    t += h[q], inc[q] = t;
  }
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
  if (!hit) {
    Z = above + __shfl_sync(0xffffffffu, off + t, 31);
    return -1;
  }
  const int src = __ffs(hit) - 1;
  float z = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (q == first) z = above + off + inc[q];
  Z = __shfl_sync(0xffffffffu, z, src);
  return 8 * src + __shfl_sync(0xffffffffu, first, src);
}

// The row pair's window band is complete: find the top-p boundaries in it,
// or queue the next band down for the sides whose boundary lies below it
// (after kMaxBands bands, an exact descent over the row); then decide.
template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void merge_window(const SParams& P, float* fh, int b, int i, char* st) {
  const int lane = threadIdx.x & 31;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  if constexpr (EBT == 2) {
    const char* parts = P.parts + pair * P.n_ch * (size_t)P.part_bytes;
    PairSt* pr = pair_st(st, P, pair);
    PairStats* ps = P.pstats + pair;
    // the row's first-pass statistics and parameters, one per lane
    uint32_t w = 0u;
    if (lane < 8) w = ld_relaxed(reinterpret_cast<const uint32_t*>(pr) + lane);
    else if (lane < 16) w = __ldcg(reinterpret_cast<const uint32_t*>(ps) + (lane - 8));
    else if (lane == 16) w = __float_as_uint(P.temperature[b]);
    else if (lane == 17) w = __float_as_uint(P.top_p[b]);
    else if (lane == 18) w = (uint32_t)(P.k ? P.k[b] : P.kmax);
    else if (lane == 19) w = i < P.kmax ? (uint32_t)P.tokens[(size_t)b * P.kmax + i] : 0u;
    const ReqScalars rs = req_scalars(P, b);
    const uint32_t wside = __shfl_sync(0xffffffffu, w, 3);
    const uint32_t lo_t = __shfl_sync(0xffffffffu, w, 4), hi_t = __shfl_sync(0xffffffffu, w, 5);
    const uint32_t lo_d = __shfl_sync(0xffffffffu, w, 6), hi_d = __shfl_sync(0xffffffffu, w, 7);
    const float Mt = __uint_as_float(__shfl_sync(0xffffffffu, w, 8));
    const float St = __uint_as_float(__shfl_sync(0xffffffffu, w, 9));
    const float Md = __uint_as_float(__shfl_sync(0xffffffffu, w, 10));
    const float Sd = __uint_as_float(__shfl_sync(0xffffffffu, w, 11));
    const float vt = __uint_as_float(__shfl_sync(0xffffffffu, w, 12));
    const float vd = __uint_as_float(__shfl_sync(0xffffffffu, w, 13));
    float above_t = __uint_as_float(__shfl_sync(0xffffffffu, w, 14));
    float above_d = __uint_as_float(__shfl_sync(0xffffffffu, w, 15));
    const float T = __uint_as_float(__shfl_sync(0xffffffffu, w, 16));
    const float top_p = __uint_as_float(__shfl_sync(0xffffffffu, w, 17));
    const int kb = (int)__shfl_sync(0xffffffffu, w, 18);
    const int y = (int)__shfl_sync(0xffffffffu, w, 19);
    const bool has_d = i < kb;
    RowP rt, rd;
    row_params<EBT, EBD, PROBS>(Mt, St, Md, Sd, has_d, T, rt, rd);
    if (lane == 0) SV_TR(31, wside, pair);
    // sides already decided in an earlier band keep their boundary in the row record
    const RowRec prev = P.rows[pair];
    if (!(wside & 1u)) rt.Dstar = prev.t.Dstar, rt.Z = prev.t.Z, rt.invZ = prev.t.invZ, rt.vstar = prev.t.vstar;
    if (has_d && !(wside & 2u))
      rd.Dstar = prev.d.Dstar, rd.Z = prev.d.Z, rd.invZ = prev.d.invZ, rd.vstar = prev.d.vstar;
    uint32_t miss = 0u;
    if (wside & 1u) {
      float Z = 0.0f;
      const int j = band_scan(P, parts, 0, hi_t, rt, top_p * rt.S, above_t, fh, Z);
      if (j >= 0) {
        const uint32_t key = hi_t - (uint32_t)j;
        rt.Dstar = rt.kmax - key, rt.Z = Z, rt.invZ = 1.0f / Z, rt.vstar = vkey_value<2>(key);
      } else {
        above_t = Z, miss |= 1u;
      }
    }
    if constexpr (EBD == 2 && !PROBS) {
      if (wside & 2u) {
        float Z = 0.0f;
        const int j = band_scan(P, parts, 1, hi_d, rd, top_p * rd.S, above_d, fh, Z);
        if (j >= 0) {
          const uint32_t key = hi_d - (uint32_t)j;
          rd.Dstar = rd.kmax - key, rd.Z = Z, rd.invZ = 1.0f / Z, rd.vstar = vkey_value<2>(key);
        } else {
          above_d = Z, miss |= 2u;
        }
      }
    }
    const uint32_t band = wside >> 8;
    if (miss && band + 1 < (uint32_t)kMaxBands && ((miss & 1u) ? lo_t : 1u) > 0u &&
        ((miss & 2u) ? lo_d : 1u) > 0u) {
      // the next band down for the sides that missed; the found side keeps
      // its boundary in the row record meanwhile
      if (lane == 0) {
        RowRec rec = prev;
        if (!(miss & 1u)) rec.t = RowSide{rt.m, rt.mz, rt.c, rt.invT, rt.Z, rt.invZ, rt.vstar, rt.Dstar};
        if (!(miss & 2u) && has_d) rec.d = RowSide{rd.m, rd.mz, rd.c, rd.invT, rd.Z, rd.invZ, rd.vstar, rd.Dstar};
        P.rows[pair] = rec;
        ps->above_t = above_t, ps->above_d = above_d;
        if (miss & 1u) pr->hi_t = lo_t - 1u, pr->lo_t = lo_t - 1u >= 255u ? lo_t - 1u - 255u : 0u;
        if (miss & 2u) pr->hi_d = lo_d - 1u, pr->lo_d = lo_d - 1u >= 255u ? lo_d - 1u - 255u : 0u;
        pr->wside = ((band + 1u) << 8) | miss;
        pr->warrive = 0u;
        __threadfence();
        queue_window(P, st, b, i, miss, pr->lo_t, pr->hi_t, pr->lo_d, pr->hi_d);
      }
      __syncwarp();
      return;
    }
    // a boundary below every band (or rounding left top_p * S out of reach):
    // the exact descent over the whole row
    if (miss & 1u) {
      const char* trow = P.target + pair * (size_t)P.t_ld * EBT;
      exact_top_p_warp<EBT, false>(trow, P.V, rt, top_p * rt.S, fh);
    }
    if (miss & 2u) {
      const char* drow = P.draft + ((size_t)b * P.kmax + i) * (size_t)P.d_ld * EBD;
      exact_top_p_warp<EBD, PROBS>(drow, P.V, rd, top_p * rd.S, fh);
    }
    if (lane == 0) {  // the depth of this nucleus guides later bands
      CallSt* cs = call_st(st);
      const float dt = (rt.m - rt.vstar) * rt.c;
      if (dt > 0.0f && dt <= FLT_MAX) atomicMax(&cs->depth_t, __float_as_uint(dt));
      if (has_d && !PROBS) {
        const float dd = (rd.m - rd.vstar) * rd.c;
        if (dd > 0.0f && dd <= FLT_MAX) atomicMax(&cs->depth_d, __float_as_uint(dd));
      }
    }
    decide_row<EBT, EBD, PROBS>(P, st, b, i, kb, y, has_d, false, rt, rd, vt, vd, rs);
  }
}

template <int EBT, int EBD, bool PROBS>
__device__ void fin_row(const SParams& P, SSmem& sm, int f, char* st) {
  const int lane = threadIdx.x & 31;
  Fin& F = sm.fin[f];
  const int b = F.b, i = F.i, c = F.c, has_d = F.has_d, kb = F.kb, y = F.y;
  const float T = F.T, top_p = F.top_p;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  char* part = P.parts + (pair * P.n_ch + c) * (size_t)P.part_bytes;
  // the consumer warps' partials, rescaled to the chunk maxima
  const bool greedy = T == 0.0f;
  const float ct = greedy ? 0.0f : kLog2e / T;
  const float invT = greedy ? 0.0f : 1.0f / T;
  const float cd = PROBS ? 1.0f : ct;
  const float4 wv = lane < kGW ? F.wp[lane] : make_float4(-INFINITY, 0.0f, PROBS ? 0.0f : -INFINITY, 0.0f);
  float Mt = wv.x, Md = wv.z;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, o));
    Md = fmaxf(Md, __shfl_xor_sync(0xffffffffu, Md, o));
  }
  float St = rescale(wv.x, wv.y, Mt, ct, greedy);
  float Sd = rescale(weight_max<PROBS>(wv.z, greedy, invT), wv.w, weight_max<PROBS>(Md, greedy, invT), cd, greedy);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    St += __shfl_xor_sync(0xffffffffu, St, o);
    Sd += __shfl_xor_sync(0xffffffffu, Sd, o);
  }
  uint32_t last = 0u;
  if (lane == 0) {
    float4* ph = reinterpret_cast<float4*>(part);
    ph[0] = make_float4(Mt, St, Md, Sd);
    ph[1] = make_float4(F.vt, F.vd, F.has_y ? 1.0f : 0.0f, 0.0f);
    mbar_arrive1(&sm.fin_empty[f]);
    __threadfence();
    last = atomicAdd(&pair_st(st, P, pair)->arrive, 1u) + 1u == (uint32_t)P.n_ch;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (lane == 0) SV_TR(21, last, pair);
  if (last) {
    __threadfence();
    merge_pass1<EBT, EBD, PROBS>(P, b, i, has_d, kb, T, top_p, y, st);
    if (lane == 0) SV_TR(22, 0, pair);
  }
}

template <int EBT, int EBD, bool PROBS>
__device__ void fin_win(const SParams& P, SSmem& sm, int f, float* fh, char* st) {
  const int lane = threadIdx.x & 31;
  Fin& F = sm.fin[f];
  const int b = F.b, i = F.i, c = F.c, win = F.win;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  char* part = P.parts + (pair * P.n_ch + c) * (size_t)P.part_bytes;
#pragma unroll
  for (int side = 0; side < 2; ++side) {
    if (win & (1 << side)) {  // bins 8l .. 8l+7 as u16, then clear them for the next use
      uint4* hs = reinterpret_cast<uint4*>(&F.hist[side][8 * lane]);
      const uint4 a = hs[0], bb = hs[1];
      hs[0] = make_uint4(0u, 0u, 0u, 0u);
      hs[1] = make_uint4(0u, 0u, 0u, 0u);
      const uint4 v = make_uint4(a.x | (a.y << 16), a.z | (a.w << 16), bb.x | (bb.y << 16), bb.z | (bb.w << 16));
      *reinterpret_cast<uint4*>(part + kPartHead + side * 512 + 16 * lane) = v;
    }
  }
  __threadfence();
  __syncwarp();
  uint32_t last = 0u;
  if (lane == 0) {
    mbar_arrive1(&sm.fin_empty[f]);
    last = atomicAdd(&pair_st(st, P, pair)->warrive, 1u) + 1u == (uint32_t)P.n_ch;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (lane == 0) SV_TR(25, last, pair);
  if (last) {
    __threadfence();
    merge_window<EBT, EBD, PROBS>(P, fh, b, i, st);
    if (lane == 0) SV_TR(26, 0, pair);
  }
}

template <int EBT, int EBD, bool PROBS>
__device__ void fin_race(const SParams& P, SSmem& sm, int f, char* st) {
  const int lane = threadIdx.x & 31;
  Fin& F = sm.fin[f];
  const int b = F.b, r = F.i, pos = F.pos;
  const uint32_t rid = F.rid;
  const float rw = F.rw, rE = F.rE;
  const int ridx = F.ridx;
  const RowRec rr = F.rr;
  __syncwarp();
  ReqSt* rq = req_st(st, b);
  uint32_t last = 0u;
  if (lane == 0) {
    mbar_arrive1(&sm.fin_empty[f]);
    if (rw > 0.0f) atomicMax(&rq->best, race_key(rw, rE, ridx));
    __threadfence();
    last = atomicAdd(&rq->race_cnt, 1u) + 1u == (uint32_t)P.n_ch;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (lane == 0) SV_TR(23, last, b);
  if (!last) return;
  __threadfence();
  unsigned long long best = 0ull;
  if (lane == 0) best = ld_relaxed64(&rq->best);
  best = __shfl_sync(0xffffffffu, best, 0);
  int token = (int)(0xFFFFFFFFu - (uint32_t)best);
  uint32_t extra = 0u;
  if ((best >> 32) == 0ull) {
    // the residual max(0, p - q) is numerically empty: draw from p with the
    // same exponentials, over the whole row (rare: read from global memory)
    extra = SV_ST_RESIDUAL_EMPTY;
    const bool greedy = rr.t.invT == 0.0f;
    RowP rt = row_p(rr.t, greedy);
    rt.kmax = vkey<EBT>(rt.m);
    const char* trow = P.target + ((size_t)b * (P.kmax + 1) + r) * (size_t)P.t_ld * EBT;
    token = race_row_warp<EBT>(trow, P.V, rt, (uint32_t)pos, rid, P.seed_lo, P.seed_hi);
  }
  if (lane == 0) {
    const unsigned long long qz = qz_mask(P, rq);
    int32_t* ot = P.out_tokens + (size_t)b * (P.kmax + 1);
    for (int j = 0; j <= P.kmax; ++j)
      ot[j] = j < r ? P.tokens[(size_t)b * P.kmax + j] : (j == r ? token : -1);
    P.accepted[b] = r;
    P.num_emitted[b] = r + 1;
    P.status[b] = qz_bits(qz, r) | extra;
    request_done(st);
    SV_TR(24, r, b);
  }
  __syncwarp();
}

template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void finisher(const SParams& P, SSmem& sm, char* st) {
  const int lane = threadIdx.x & 31;
  const int w = ((int)threadIdx.x >> 5) - kFinisherWarp;  // 0 .. kFW-1
  float* fh = sm.fh[w];
  uint32_t ph = 0u;
  for (int f = w;; f = f + kFW >= kNF ? f + kFW - kNF : f + kFW) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_ns(&sm.fin_full[f], (ph >> f) & 1u, P.err, kFinWaitNs, 512u);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();  // lane 0's acquire orders the other lanes' reads of the slot too
    ph ^= 1u << f;
    if (!ok) break;
    const int kind = sm.fin[f].kind;
    if (lane == 0) SV_TR(20, kind, f);
    if (kind == kEnd) break;
    if (kind == kRowItem) {
      fin_row<EBT, EBD, PROBS>(P, sm, f, st);
    } else if (kind == kWinItem) {
      fin_win<EBT, EBD, PROBS>(P, sm, f, fh, st);
    } else if (kind == kRaceItem) {
      fin_race<EBT, EBD, PROBS>(P, sm, f, st);
    } else {
      const int b = sm.fin[f].b;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive1(&sm.fin_empty[f]);
        ReqSt* rq = req_st(st, b);
        if (atomicCAS(&rq->resolved, 0u, 1u) == 0u) {
          bad_outputs(P, b, SV_ST_BAD_INPUT);
          __threadfence();
          atomicAdd(&call_st(st)->cnt, kResolvedOne);
          request_done(st);
        }
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int EBT, int EBD, bool PROBS>
__global__ void __launch_bounds__(kAllThreads, 1) stream_kernel(const SParams P) {
  constexpr int NS = num_stages<EBT, EBD>();
  __shared__ SSmem sm;
  extern __shared__ __align__(128) char dyn[];
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_wait();     // whatever ran before (the logits' producer, an earlier call) has finished
  pdl_trigger();  // the next kernel (e.g. the commit) may be scheduled and wait in its own pdl_wait
  const uint32_t par = *reinterpret_cast<volatile const uint32_t*>(&P.hdr->parity) & 1u;
  char* st = P.state[par];
  {  // zero the half the next call uses
    uint32_t* other = reinterpret_cast<uint32_t*>(P.state[par ^ 1u]);
    for (size_t w = (size_t)blockIdx.x * kAllThreads + tid; w < P.state_words;
         w += (size_t)gridDim.x * kAllThreads)
      other[w] = 0u;
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init_n(&sm.full[s], 1), mbar_init_n(&sm.empty[s], kGW);
    for (int f = 0; f < kNF; ++f) mbar_init_n(&sm.fin_full[f], kGW), mbar_init_n(&sm.fin_empty[f], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  for (int j = tid; j < kNF * 2 * kBins; j += kAllThreads)
    (&sm.fin[j / (2 * kBins)].hist[0][0])[j % (2 * kBins)] = 0u;
#ifdef SV_TRACE
  if (tid == 0) trace_slot() = 0u;
#endif
  __syncthreads();
  if (warp == kProducerWarp) producer<EBT, EBD, PROBS>(P, sm, dyn, st);
  else if (warp >= kFinisherWarp) finisher<EBT, EBD, PROBS>(P, sm, st);
  else consumer<EBT, EBD, PROBS>(P, sm, dyn);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&P.hdr->exit_cnt, 1u);
    if (d + 1u == gridDim.x) {
      P.hdr->ticket = 0u;
      P.hdr->dticket = 0u;
      P.hdr->exit_cnt = 0u;
      // the next call's first bands start from this call's deepest nuclei
      const uint32_t dt = ld_relaxed(&call_st(st)->depth_t), dd = ld_relaxed(&call_st(st)->depth_d);
      if (dt) P.hdr->depth_t = dt;
      if (dd) P.hdr->depth_d = dd;
      __threadfence();
      atomicAdd(&P.hdr->parity, 1u);
    }
  }
}

// ---------------------------------------------------------------------------
// Normalised rows (debug output): one block per (row pair, chunk) writes
// prob(v) of every element of the decided rows of the call just finished.
// ---------------------------------------------------------------------------
template <int EBT, int EBD, bool PROBS>
__global__ void __launch_bounds__(256) stream_probs_kernel(const SParams P, float* probs_p,
                                                           float* probs_q) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  const uint32_t par = (*reinterpret_cast<volatile const uint32_t*>(&P.hdr->parity) & 1u) ^ 1u;
  char* st = P.state[par];
  const size_t pair = blockIdx.x;
  const int b = (int)(pair / (size_t)(P.kmax + 1)), i = (int)(pair % (size_t)(P.kmax + 1));
  const uint32_t state = ld_relaxed(&pair_st(st, P, pair)->state);
  if (state == 0u || state == SV_ROW_INVALID) return;
  const RowRec rr = P.rows[pair];
  const bool greedy = rr.t.invT == 0.0f;
  RowP rt = row_p(rr.t, greedy), rd = row_p(rr.d, greedy);
  rt.kmax = vkey<EBT>(rt.m);
  rd.kmax = vkey<EBD>(rd.m);
  const int kb = P.k ? P.k[b] : P.kmax;
  const int x0 = blockIdx.y * CH, x1 = min(P.V, x0 + CH);
  const char* trow = P.target + pair * (size_t)P.t_ld * EBT;
  for (int x = x0 + threadIdx.x; x < x1; x += blockDim.x)
    probs_p[pair * (size_t)P.V + x] = prob<EBT, false>(row_value<EBT>(trow, x), rt);
  if (probs_q && i < kb) {
    const size_t drw = (size_t)b * P.kmax + i;
    const char* drow = P.draft + drw * (size_t)P.d_ld * EBD;
    for (int x = x0 + threadIdx.x; x < x1; x += blockDim.x)
      probs_q[drw * (size_t)P.V + x] = prob<EBD, PROBS>(row_value<EBD>(drow, x), rd);
  }
}

}  // namespace stream
}  // namespace sv
