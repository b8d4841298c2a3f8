#pragma once
// Streaming verification kernel: producer, consumers and finishers, the
// row-pair combine and the request resolution (see stream_kernel.cuh).
#include "stream_kernel.cuh"

namespace sv {
namespace stream {

// Barrier among the consumer warps that also ORs a per-thread flag.
__device__ __forceinline__ bool cbar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{.reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q;}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kCT)
      : "memory");
  return r != 0u;
}

// ---------------------------------------------------------------------------
// Request state (finisher lane 0 writes, producers read)
// ---------------------------------------------------------------------------
constexpr unsigned long long kResolvedOne = 1ull << 32;  // CallSt::cnt, resolved count

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

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
  if (sf < 0) sf = (int)ld_relaxed(&pair_st(st, P.B, (size_t)b * (P.kmax + 1) + f)->state);
  if (sf == SV_ROW_REJECTED || sf == SV_ROW_BONUS) {
    // one atomic counts the resolution and claims the race slot: a waiter that
    // sees every request resolved also sees every slot claimed
    const uint32_t q = (uint32_t)atomicAdd(&cs->cnt, kResolvedOne | 1ull);
    Slot* sl = slot_st(st, P.B, (int)q);
    sl->b = (uint32_t)b;
    sl->row = (uint32_t)f;
    sl->kind = sf == SV_ROW_REJECTED ? kRaceResidual : kRaceBonus;
    st_release(&sl->ready, 1u);
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

// ---------------------------------------------------------------------------
// Producer warp
// ---------------------------------------------------------------------------
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
  const uint32_t tt = (uint32_t)target * (uint32_t)P.n_ch;
  uint32_t t = 0u;
  if (lane == 0) {
    const uint32_t old = atomicMax(&P.hdr->ticket, tt + 1u);
    t = old <= tt ? tt : atomicAdd(&P.hdr->ticket, 1u);
  }
  return __shfl_sync(0xffffffffu, t, 0);
}

// A waiter gave up on a race slot: requests never resolved are reported as
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

template <int EBT, int EBD, bool PROBS>
__device__ void producer(const SParams& P, SSmem& sm, char* dyn, char* st) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int NS = num_stages<EBT, EBD>();
  constexpr int SB = stage_bytes<EBT, EBD>();
  const int lane = threadIdx.x & 31;
  CallSt* cs = call_st(st);
  uint32_t used = 0u, eph = 0u;  // per stage: used once / parity of its next empty phase
  int s = 0;
  // Two tickets in hand: the next one's atomic is in flight while the current
  // one is settled.  The smaller is always settled first, so a static ticket
  // is never held while waiting on a race slot.
  uint32_t t = take_ticket(P), tn = take_ticket(P);
  for (;;) {
    SHdr h;
    h.kind = kEnd;
    h.b = h.i = h.c = 0;
    h.x0 = h.n = h.has_d = h.kb = 0;
    h.T = 0.0f, h.top_p = 1.0f;
    h.race = 0, h.pos = 0, h.rid = 0u, h.y = 0;
    // ------------------------------------------------------------ settle
    for (;;) {
      if (tn < t) {
        const uint32_t x = t;
        t = tn, tn = x;
      }
      if (t < P.n_static) {
        const int R = (int)(t / (uint32_t)P.n_ch);
        const int c = (int)(t - (uint32_t)R * (uint32_t)P.n_ch);
        const int i = R / P.B, b = R - i * P.B;
        // the request's parameters, one per lane, in one round trip
        int iv = 0;
        float fv = 0.0f;
        if (lane == 0) iv = P.k ? P.k[b] : P.kmax;
        if (lane == 1) iv = P.max_new ? P.max_new[b] : 0x7FFFFFFF;
        if (lane == 2) iv = (i > 0 && !(P.flags & SV_FLAG_NO_SKIP)) ? first_nonacc(P, st, b) : (int)kNA;
        if (lane == 3) fv = P.temperature[b];
        if (lane == 4) fv = P.top_p ? P.top_p[b] : 1.0f;
        if (lane == 5 && i < P.kmax) iv = P.tokens[(size_t)b * P.kmax + i];
        const int kb = __shfl_sync(0xffffffffu, iv, 0);
        const int cap = __shfl_sync(0xffffffffu, iv, 1);
        const int fna = __shfl_sync(0xffffffffu, iv, 2);
        const float T = __shfl_sync(0xffffffffu, fv, 3);
        const float tp = __shfl_sync(0xffffffffu, fv, 4);
        const int y = __shfl_sync(0xffffffffu, iv, 5);
        const int what = interest_of(P, i, kb, cap, fna);
        if (what == 1 || (what == 2 && c == 0)) {
          h.kind = what == 1 ? kRowItem : kBadItem;
          h.b = b, h.i = i, h.c = c;
          if (what == 1) {
            h.kb = kb;
            h.has_d = i < kb;
            h.x0 = c * CH;
            h.n = min(CH, P.V - h.x0);
            h.T = T;
            h.top_p = tp;
            h.y = h.has_d ? y : 0;
          }
          break;
        }
        t = jump_ticket(P, st, R);
        if (lane == 0) SV_TR(3, R, t);
        continue;
      }
      const uint32_t rt = t - P.n_static;
      const int q = (int)(rt / (uint32_t)P.n_ch);
      const int part = (int)(rt - (uint32_t)q * (uint32_t)P.n_ch);
      if (q >= P.B) break;  // END
      Slot* sl = slot_st(st, P.B, q);
      bool go = false;
      const unsigned long long t0 = gtimer();
      for (int spins = 0;; ++spins) {
        if (ld_acquire(&sl->ready)) {
          go = true;
          break;
        }
        const unsigned long long c = ld_acquire64(&cs->cnt);
        if ((uint32_t)(c >> 32) >= (uint32_t)P.B && (uint32_t)c <= (uint32_t)q) break;
        if (gtimer() - t0 > P.slot_wait_ns) {
          timeout_sweep(P, st);
          break;
        }
        __nanosleep(spins < 64 ? 64 : 256);
      }
      if (!go) break;  // END
      int iv = 0;
      if (lane == 0) iv = (int)ld_relaxed(&sl->b);
      if (lane == 1) iv = (int)ld_relaxed(&sl->row);
      if (lane == 2) iv = (int)ld_relaxed(&sl->kind);
      const int b = __shfl_sync(0xffffffffu, iv, 0);
      const int r = __shfl_sync(0xffffffffu, iv, 1);
      h.kind = kRaceItem;
      h.b = b, h.i = r, h.c = part;
      h.race = __shfl_sync(0xffffffffu, iv, 2);
      h.has_d = h.race == kRaceResidual;
      h.x0 = part * CH;
      h.n = min(CH, P.V - h.x0);
      int pv = 0;
      if (lane == 0) pv = P.seq_len ? P.seq_len[b] : 0;
      if (lane == 1) pv = P.request_id ? (int)P.request_id[b] : b;
      h.pos = __shfl_sync(0xffffffffu, pv, 0) + 1 + r;
      h.rid = (uint32_t)__shfl_sync(0xffffffffu, pv, 1);
      break;
    }
    if (lane == 0) SV_TR(1, (h.kind << 20) | (h.i << 12) | h.c, h.b);
    // ------------------------------------------------ wait for the stage
    if (used & (1u << s)) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait_ns(&sm.empty[s], (eph >> s) & 1u, P.err, kStageWaitNs, 256u);
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
    }
    __syncwarp();
    if (lane == 0) {
      if (h.kind == kRowItem || h.kind == kRaceItem) {
        char* sT = dyn + (size_t)s * SB;
        char* sD = sT + (size_t)CH * EBT;
        const uint32_t bt = (uint32_t)((h.n * EBT + 15) & ~15);
        const uint32_t bd = h.has_d ? (uint32_t)((h.n * EBD + 15) & ~15) : 0u;
        const char* trow = P.target + ((size_t)h.b * (P.kmax + 1) + h.i) * (size_t)P.t_ld * EBT;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(&sm.full[s], bt + bd);
        bulk_g2s(sT, trow + (size_t)h.x0 * EBT, bt, &sm.full[s]);
        if (h.has_d) {
          const char* drow = P.draft + ((size_t)h.b * P.kmax + h.i) * (size_t)P.d_ld * EBD;
          bulk_g2s(sD, drow + (size_t)h.x0 * EBD, bd, &sm.full[s]);
        }
      } else {
        mbar_arrive1(&sm.full[s]);
      }
    }
    if (lane == 0) SV_TR(2, s, t);
    if (h.kind == kEnd) break;
    s = s + 1 == NS ? 0 : s + 1;
    t = tn, tn = take_ticket(P);
  }
}

// ---------------------------------------------------------------------------
// Consumers
// ---------------------------------------------------------------------------
// Window floor: the bf16 key `depth` log2 units below the reference key (at
// most 255 keys below it); thr2 is its value as a packed pair.
__device__ __forceinline__ void window_floor(uint32_t ref, float depth, float c, uint32_t& fk,
                                             uint32_t& thr2) {
  const float D = depth > 0.0f ? depth + kDepthMargin
                              : (SV_STREAM_DEPTH0 > 0.0f ? SV_STREAM_DEPTH0 : INFINITY);
  const float fv = vkey_value<2>(ref) - D / c;
  uint32_t k = 0u;
  if (fv > -INFINITY) k = key16(__uint_as_float(bf16_pair_of(fv) << 16));
  const uint32_t lo = ref >= 255u ? ref - 255u : 0u;
  if (k < lo) k = lo;
  if (k > ref) k = ref;
  fk = k;
  const uint32_t hb = __float_as_uint(vkey_value<2>(k)) >> 16;
  thr2 = hb | (hb << 16);
}

// Window counts of one bf16 chunk into ring bins (-key) & 255 of `hist`.
__device__ __forceinline__ void window_chunk(const char* s, const SliceIter& it, uint32_t thr2,
                                             uint32_t* hist, uint8_t* wb) {
  uint32_t lo = 0u, hi = 0u;
  int cnt = 0;
#pragma unroll kStreamUnroll
  for (int j = 0; j < kMaxBlk; ++j) {
    if (j < it.nblk) {
      const uint4 g = load_group_bf16(s, it, j);
      const uint32_t m = window_bits_bf16(g, thr2, it.x(j), it.x1);
      cnt += __popc(m);
      if (j < 4) lo |= m << (8 * j);
      else hi |= m << (8 * (j - 4));
    }
  }
  window_commit_bf16(s, 0u, lo, hi, cnt, it, hist, wb);
}

template <int EBT, int EBD, bool PROBS>
__device__ void process_row(const SParams& P, SSmem& sm, const SHdr& h, int s, int f, const char* sT,
                            const char* sD, char* st) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int GPT = CH / kGroup / kCT;
  const int ctid = threadIdx.x, lane = ctid & 31, warp = ctid >> 5;
  const bool has_d = h.has_d;
  const float T = h.T, top_p = h.top_p;
  const bool greedy = T == 0.0f;
  const bool pok = row_params_ok(T, top_p);
  const float ct = greedy ? 0.0f : kLog2e / T;
  const float invT = greedy ? 0.0f : 1.0f / T;
  const float cd = PROBS ? 1.0f : ct;
  SliceIter it;
  it.x0 = h.x0, it.x1 = h.x0 + h.n, it.nblk = GPT, it.V = P.V;
  it.stride = kCT * kGroup, it.tid = (int)threadIdx.x;
  const size_t pair = (size_t)h.b * (P.kmax + 1) + h.i;
  PairSt* ps = pair_st(st, P.B, pair);
  Fin& F = sm.fin[f];

  // ---------------------------------------------------------- maxima
  uint32_t mt2 = 0xFF80FF80u, md2 = 0xFF80FF80u;
  float rmt = -INFINITY, rmd = PROBS ? 0.0f : -INFINITY;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int x = it.x(j);
    if (x < it.x1) {
      Grp<EBT> g;
      lds_group<EBT, false>(g, sT, it.x0, x, it.x1);
      max_group<EBT>(g, mt2, rmt);
      if (has_d) {
        Grp<EBD> q;
        lds_group<EBD, PROBS>(q, sD, it.x0, x, it.x1);
        max_group<EBD>(q, md2, rmd);
      }
    }
  }
  float mt = max_value<EBT>(mt2, rmt), md = max_value<EBD>(md2, rmd);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, o));
  }
  if (lane == 0) sm.red[warp][0] = mt, sm.red[warp][1] = md;
  cbar();
  if (ctid == 0) SV_TR(11, 0, 0);
  float Mt = -INFINITY, Md = PROBS ? 0.0f : -INFINITY;
#pragma unroll
  for (int w = 0; w < kCW; ++w) Mt = fmaxf(Mt, sm.red[w][0]), Md = fmaxf(Md, sm.red[w][1]);
  const float Mzd = weight_max<PROBS>(Md, greedy, invT);
  const bool topp = !greedy && pok && top_p < 1.0f && P.hist;
  const bool win_t = EBT == 2 && topp;
  const bool win_d = EBD == 2 && !PROBS && topp && has_d;
  // Thread 0 reads the window hints (largest chunk maxima published for this
  // row pair, deepest nucleus of the call) and shares them through shared
  // memory: every thread must use the same window floor.  The loads are
  // issued now and consumed after the sums, so their latency hides.
  uint32_t hv[4] = {0u, 0u, 0u, 0u};
  if (ctid == 0 && (win_t || win_d)) {
    if (win_t) atomicMax(&ps->tkey, key16(Mt));
    if (win_d) atomicMax(&ps->dkey, key16(Md));
    if (win_t) hv[0] = ld_relaxed(&ps->tkey), hv[2] = ld_relaxed(&call_st(st)->depth_t);
    if (win_d) hv[1] = ld_relaxed(&ps->dkey), hv[3] = ld_relaxed(&call_st(st)->depth_d);
  }
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
  }

  // ------------------------------------------------- weight sums
  float sumt = 0.0f, sumd = 0.0f;
#pragma unroll kStreamUnroll
  for (int j = 0; j < GPT; ++j) {
    const int x = it.x(j);
    if (x < it.x1) {
      Grp<EBT> g;
      lds_group<EBT, false>(g, sT, it.x0, x, it.x1);
      sumt += sum_group<EBT, false>(g, greedy, Mt, ct, invT);
      if (has_d) {
        Grp<EBD> q;
        lds_group<EBD, PROBS>(q, sD, it.x0, x, it.x1);
        sumd += sum_group<EBD, PROBS>(q, greedy, Mzd, cd, invT);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    sumt += __shfl_xor_sync(0xffffffffu, sumt, o);
    sumd += __shfl_xor_sync(0xffffffffu, sumd, o);
  }
  if (lane == 0) sm.red[warp][2] = sumt, sm.red[warp][3] = sumd;
  if (ctid == 0) sm.hint[0] = hv[0], sm.hint[1] = hv[1], sm.hint[2] = hv[2], sm.hint[3] = hv[3];
  cbar();
  if (ctid == 0) SV_TR(12, 0, 0);

  // ------------------------------------------ top-p window counts
  uint32_t ref_t = 0u, flo_t = 0xFFFFFFFFu, ref_d = 0u, flo_d = 0xFFFFFFFFu;
  if constexpr (EBT == 2) {
    if (win_t) {
      uint32_t thr2;
      ref_t = max(key16(Mt), sm.hint[0]);
      window_floor(ref_t, __uint_as_float(sm.hint[2]), ct, flo_t, thr2);
      window_chunk(sT, it, thr2, F.hist[0], sm.wb.bin[warp]);
    }
  }
  if constexpr (EBD == 2 && !PROBS) {
    if (win_d) {
      uint32_t thr2;
      ref_d = max(key16(Md), sm.hint[1]);
      window_floor(ref_d, __uint_as_float(sm.hint[3]), cd, flo_d, thr2);
      window_chunk(sD, it, thr2, F.hist[1], sm.wb.bin[warp]);
    }
  }
  release_stage(sm, s);

  // ---------------------------------------------- hand-off: each warp
  // arrives once its window counts are in; thread 0 writes the fields first
  if (ctid == 0) {
    float St = 0.0f, Sd = 0.0f;
    for (int w = 0; w < kCW; ++w) St += sm.red[w][2], Sd += sm.red[w][3];
    F.kind = kRowItem, F.b = h.b, F.i = h.i, F.c = h.c;
    F.has_d = h.has_d, F.kb = h.kb, F.T = T, F.top_p = top_p, F.y = h.y;
    F.Mt = Mt, F.St = St, F.Md = Md, F.Sd = Sd;
    F.ref_t = ref_t, F.flo_t = flo_t, F.ref_d = ref_d, F.flo_d = flo_d;
    F.win = (win_t ? 1 : 0) | (win_d ? 2 : 0);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive1(&sm.fin_full[f]);
  if (ctid == 0) SV_TR(13, f, 0);
}

template <int EBT, int EBD, bool PROBS>
__device__ void process_race(const SParams& P, SSmem& sm, const SHdr& h, int s, int f, const char* sT,
                             const char* sD) {
  constexpr int GPT = chunk_elems<EBT, EBD>() / kGroup / kCT;
  const int ctid = threadIdx.x, lane = ctid & 31, warp = ctid >> 5;
  const RowRec rr = h.rr;
  const bool greedy = rr.t.invT == 0.0f;
  RowP rt = row_p(rr.t, greedy), rd = row_p(rr.d, greedy);
  rt.kmax = vkey<EBT>(rt.m);
  rd.kmax = vkey<EBD>(rd.m);
  const bool residual = h.race == kRaceResidual;
  SliceIter it;
  it.x0 = h.x0, it.x1 = h.x0 + h.n, it.nblk = GPT, it.V = P.V;
  it.stride = kCT * kGroup, it.tid = (int)threadIdx.x;
  RacePart best = {0.0f, 1.0f, 0x7FFFFFFF};
  race_slice<EBT, EBD, PROBS>(sT, sD, it, residual, rt, rd, (uint32_t)h.pos, h.rid, P.seed_lo, P.seed_hi,
                              sm.wb.idx[warp], best);
  release_stage(sm, s);
  warp_race(best.w, best.E, best.idx);
  if (lane == 0) sm.rp[warp] = best;
  cbar();
  if (ctid == 0) {
    RacePart o = sm.rp[0];
    for (int w = 1; w < kCW; ++w)
      if (better(sm.rp[w].w, sm.rp[w].E, sm.rp[w].idx, o.w, o.E, o.idx)) o = sm.rp[w];
    Fin& F = sm.fin[f];
    F.kind = kRaceItem, F.b = h.b, F.i = h.i, F.c = h.c;
    F.race = h.race, F.pos = h.pos, F.rid = h.rid;
    F.rw = o.w, F.rE = o.E, F.ridx = o.idx;
    F.rr = h.rr;
    mbar_arrive_n(&sm.fin_full[f], kCW);
  }
}

template <int EBT, int EBD, bool PROBS>
__device__ void consumer(const SParams& P, SSmem& sm, char* dyn, char* st) {
  constexpr int CH = chunk_elems<EBT, EBD>();
  constexpr int NS = num_stages<EBT, EBD>();
  constexpr int SB = stage_bytes<EBT, EBD>();
  uint32_t fph = 0u, fused = 0u, feph = 0u;
  int s = 0, f = 0;
  for (;;) {
    // Thread 0 waits for the stage's data and for a free hand-off slot; the
    // other consumer warps wait in the barrier (issuing nothing), which also
    // carries the outcome, so every consumer thread takes the same path (a
    // wait that did not complete in time ends this CTA's work).  The barrier
    // orders the stage's contents, seen complete by thread 0, before every
    // thread's reads.
    bool ok = true;
    if (threadIdx.x == 0) {
      ok = mbar_wait_ns(&sm.full[s], (fph >> s) & 1u, P.err, kStageWaitNs, 64u);
      if (fused & (1u << f))
        ok = mbar_wait_ns(&sm.fin_empty[f], (feph >> f) & 1u, P.err, kStageWaitNs, 64u) && ok;
    }
    fph ^= 1u << s;
    if (fused & (1u << f)) feph ^= 1u << f;
    fused |= 1u << f;
    const bool bad = cbar_or(!ok);
    const SHdr h = sm.hdr[s];
    if (threadIdx.x == 0) SV_TR(10, h.kind, (h.b << 8) | (h.i << 4) | h.c);
    if (bad || h.kind == kEnd) {
      if (threadIdx.x == 0) {  // tell every finisher to stop
        for (int w = 0; w < kFW; ++w) {
          if (w > 0) {
            f = f + 1 == kNF ? 0 : f + 1;
            if (fused & (1u << f)) {
              (void)mbar_wait_ns(&sm.fin_empty[f], (feph >> f) & 1u, P.err, kStageWaitNs);
              feph ^= 1u << f;
            }
            fused |= 1u << f;
          }
          sm.fin[f].kind = kEnd;
          mbar_arrive_n(&sm.fin_full[f], kCW);
        }
      }
      break;
    }
    const char* sT = dyn + (size_t)s * SB;
    const char* sD = sT + (size_t)CH * EBT;
    if (h.kind == kRowItem) {
      process_row<EBT, EBD, PROBS>(P, sm, h, s, f, sT, sD, st);
    } else if (h.kind == kRaceItem) {
      process_race<EBT, EBD, PROBS>(P, sm, h, s, f, sT, sD);
    } else {  // a bad request's report
      release_stage(sm, s);
      if (threadIdx.x == 0) {
        Fin& F = sm.fin[f];
        F.kind = kBadItem, F.b = h.b;
        mbar_arrive_n(&sm.fin_full[f], kCW);
      }
    }
    s = s + 1 == NS ? 0 : s + 1;
    f = f + 1 == kNF ? 0 : f + 1;
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

template <int EBT, int EBD, bool PROBS>
__device__ __noinline__ void combine_warp(const SParams& P, float* fh, int b, int i, int has_d, int kb,
                                          float T, float top_p, int win, int y, char* st) {
  const int lane = threadIdx.x & 31;
  // the request's scalars, one per lane, loaded together with the headers
  int rv = 0;
  if (lane == 0) rv = P.seq_len ? P.seq_len[b] : 0;
  if (lane == 1) rv = P.request_id ? (int)P.request_id[b] : b;
  if (lane == 2) rv = P.eos ? P.eos[b] : -1;
  if (lane == 3) rv = P.max_new ? P.max_new[b] : 0x7FFFFFFF;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  const char* parts = P.parts + pair * P.n_ch * (size_t)P.part_bytes;
  const bool greedy = T == 0.0f;
  const bool pok = row_params_ok(T, top_p);
  const float ct = greedy ? 0.0f : kLog2e / T;
  const float invT = greedy ? 0.0f : 1.0f / T;
  const float cd = PROBS ? 1.0f : ct;
  // chunk c's header on lane c
  PartHdr ht = {-INFINITY, 0.0f, 0u, 0u}, hd = {PROBS ? 0.0f : -INFINITY, 0.0f, 0u, 0u};
  float4 hv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (lane < P.n_ch) {
    const float4* p = reinterpret_cast<const float4*>(parts + (size_t)lane * P.part_bytes);
    const float4 a = __ldcg(p), d = __ldcg(p + 1);
    hv = __ldcg(p + 2);
    ht = PartHdr{a.x, a.y, __float_as_uint(a.z), __float_as_uint(a.w)};
    if (has_d) hd = PartHdr{d.x, d.y, __float_as_uint(d.z), __float_as_uint(d.w)};
  }
  RowP rt, rd;
  rt.greedy = rd.greedy = greedy;
  {
    float M = ht.m;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = rescale(ht.m, ht.S, M, ct, greedy);
#pragma unroll
    for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    rt.m = rt.mz = M, rt.S = S;
  }
  if (has_d) {
    float M = hd.m;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float mz = weight_max<PROBS>(hd.m, greedy, invT), Mz = weight_max<PROBS>(M, greedy, invT);
    float S = rescale(mz, hd.S, Mz, cd, greedy);
#pragma unroll
    for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    rd.m = M, rd.mz = Mz, rd.S = S;
  } else {
    rd.m = rd.mz = PROBS ? 0.0f : -INFINITY, rd.S = 1.0f;
  }
  rt.c = ct, rt.invT = invT, rt.kmax = vkey<EBT>(rt.m), rt.Dstar = kNoFilter, rt.vstar = -INFINITY;
  rt.Z = rt.S, rt.invZ = 1.0f / rt.S;
  rd.c = cd, rd.invT = invT, rd.kmax = vkey<EBD>(rd.m), rd.Dstar = kNoFilter;
  rd.vstar = PROBS ? 0.0f : -INFINITY;
  rd.Z = rd.S, rd.invZ = 1.0f / rd.S;

  if (lane == 0) SV_TR(30, 0, pair);
  // the accept-test operands from the chunk that holds the proposal
  const uint32_t ym = __ballot_sync(0xffffffffu, lane < P.n_ch && hv.z != 0.0f);
  const int ysrc = ym ? __ffs(ym) - 1 : 0;
  const float vt = __shfl_sync(0xffffffffu, hv.x, ysrc), vd = __shfl_sync(0xffffffffu, hv.y, ysrc);
  const bool y_ok = !has_d || (y >= 0 && y < P.V && ym != 0u);
  const int r_seq = __shfl_sync(0xffffffffu, rv, 0), r_rid = __shfl_sync(0xffffffffu, rv, 1);
  const int r_eos = __shfl_sync(0xffffffffu, rv, 2), r_cap = __shfl_sync(0xffffffffu, rv, 3);
  const bool bad_t = !(rt.S >= 1.0f && rt.S <= FLT_MAX) || !(rt.m <= FLT_MAX) || rt.m == -INFINITY;
  const bool bad_d = has_d && (!(rd.S >= 1.0f && rd.S <= FLT_MAX) || !(rd.m <= FLT_MAX) ||
                               (PROBS ? !(rd.m > 0.0f) : rd.m == -INFINITY));
  const bool row_bad = bad_t || bad_d || !pok || !y_ok;
  const char* trow = P.target + pair * (size_t)P.t_ld * EBT;
  const char* drow = has_d ? P.draft + ((size_t)b * P.kmax + i) * (size_t)P.d_ld * EBD : nullptr;

  // ------------------------------------------------------------ top-p
  if (!row_bad && !greedy && top_p < 1.0f) {
    bool need_t = true;
    if constexpr (EBT == 2) {
      if (win & 1) {
        uint32_t F = lane < P.n_ch ? ht.floor : 0u;
#pragma unroll
        for (int o = 16; o; o >>= 1) F = max(F, __shfl_xor_sync(0xffffffffu, F, o));
        const uint32_t K = key16(rt.m);
        float Z = 0.0f;
        const int j = window_boundary(P, parts, 0, ht.ref, K, F, rt, top_p * rt.S, fh, Z);
        if (j >= 0) {
          need_t = false;
          rt.Dstar = (uint32_t)j, rt.Z = Z, rt.invZ = 1.0f / Z, rt.vstar = vkey_value<2>(K - (uint32_t)j);
        }
      }
    }
    if (lane == 0) SV_TR(31, need_t, pair);
    if (need_t) exact_top_p_warp<EBT, false>(trow, P.V, rt, top_p * rt.S, fh);
    if (has_d) {
      bool need_d = true;
      if constexpr (EBD == 2 && !PROBS) {
        if (win & 2) {
          uint32_t F = lane < P.n_ch ? hd.floor : 0u;
#pragma unroll
          for (int o = 16; o; o >>= 1) F = max(F, __shfl_xor_sync(0xffffffffu, F, o));
          const uint32_t K = key16(rd.m);
          float Z = 0.0f;
          const int j = window_boundary(P, parts, 1, hd.ref, K, F, rd, top_p * rd.S, fh, Z);
          if (j >= 0) {
            need_d = false;
            rd.Dstar = (uint32_t)j, rd.Z = Z, rd.invZ = 1.0f / Z, rd.vstar = vkey_value<2>(K - (uint32_t)j);
          }
        }
      }
      if (lane == 0) SV_TR(32, need_d, pair);
      if (need_d) exact_top_p_warp<EBD, PROBS>(drow, P.V, rd, top_p * rd.S, fh);
    }
    if (lane == 0) {  // the depth of this nucleus guides later windows
      const float dt = (rt.m - rt.vstar) * rt.c;
      if (dt > 0.0f && dt <= FLT_MAX) atomicMax(&call_st(st)->depth_t, __float_as_uint(dt));
      if (has_d && !PROBS) {
        const float dd = (rd.m - rd.vstar) * rd.c;
        if (dd > 0.0f && dd <= FLT_MAX) atomicMax(&call_st(st)->depth_d, __float_as_uint(dd));
      }
    }
  }

  // ------------------------------------------------ accept test, publish
  if (lane == 0) {
    int state;
    bool qzero = false;
    float p_y = 0.0f, q_y = 0.0f, u = 0.0f;
    if (row_bad) {
      state = SV_ROW_INVALID;
    } else if (has_d) {
      p_y = prob<EBT, false>(vt, rt);
      q_y = prob<EBD, PROBS>(vd, rd);
      const int pos = r_seq + 1 + i;
      u = uniform_from_bits(
          philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)r_rid, 1u), P.seed_lo, P.seed_hi).x);
      qzero = q_y == 0.0f;
      state = (u * q_y < p_y) ? SV_ROW_ACCEPTED : SV_ROW_REJECTED;
      if (state == SV_ROW_ACCEPTED) {
        if ((r_eos >= 0 && y == r_eos) || (r_cap <= kb && i == r_cap - 1)) state = SV_ROW_TERMINAL;
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
      d.p_kept = greedy || rt.Dstar == kNoFilter ? 1.0f : rt.Z / rt.S;
      d.q_kept = !has_d || greedy || rd.Dstar == kNoFilter ? 1.0f : rd.Z / rd.S;
      d.state = state;
      d.p_thr_key = rt.Dstar == kNoFilter ? -1 : (int32_t)(rt.kmax - rt.Dstar);
      d.q_thr_key = (!has_d || rd.Dstar == kNoFilter) ? -1 : (int32_t)(rd.kmax - rd.Dstar);
      P.debug[pair] = d;
    }
    st_relaxed(&pair_st(st, P.B, pair)->state, (uint32_t)state);
    SV_TR(33, state, pair);
    const bool withhold = (P.flags & SV_FLAG_TEST_WITHHOLD) && pair == 0;
    if (!withhold) publish(P, st, b, i, state, qzero);
  }
  __syncwarp();
}

template <int EBT, int EBD, bool PROBS>
__device__ void fin_row(const SParams& P, SSmem& sm, int f, float* fh, char* st) {
  const int lane = threadIdx.x & 31;
  Fin& F = sm.fin[f];
  const int b = F.b, i = F.i, c = F.c, has_d = F.has_d, kb = F.kb, win = F.win, y = F.y;
  const float T = F.T, top_p = F.top_p;
  const size_t pair = (size_t)b * (P.kmax + 1) + i;
  char* part = P.parts + (pair * P.n_ch + c) * (size_t)P.part_bytes;
  if (lane == 0) {
    float4* ph = reinterpret_cast<float4*>(part);
    ph[0] = make_float4(F.Mt, F.St, __uint_as_float(F.ref_t), __uint_as_float(F.flo_t));
    ph[1] = make_float4(F.Md, F.Sd, __uint_as_float(F.ref_d), __uint_as_float(F.flo_d));
    ph[2] = make_float4(F.vt, F.vd, F.has_y ? 1.0f : 0.0f, 0.0f);
  }
#pragma unroll
  for (int side = 0; side < 2; ++side) {
    if (win & (1 << side)) {  // ring bins 8l .. 8l+7 as u16, then clear them for the next use
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
    last = atomicAdd(&pair_st(st, P.B, pair)->arrive, 1u) + 1u == (uint32_t)P.n_ch;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (lane == 0) SV_TR(21, last, pair);
  if (last) {
    __threadfence();
    combine_warp<EBT, EBD, PROBS>(P, fh, b, i, has_d, kb, T, top_p, win, y, st);
    if (lane == 0) SV_TR(22, 0, pair);
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
__device__ void finisher(const SParams& P, SSmem& sm, char* st) {
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
      fin_row<EBT, EBD, PROBS>(P, sm, f, fh, st);
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
    for (int s = 0; s < NS; ++s) mbar_init_n(&sm.full[s], 1), mbar_init_n(&sm.empty[s], kCW);
    for (int f = 0; f < kNF; ++f) mbar_init_n(&sm.fin_full[f], kCW), mbar_init_n(&sm.fin_empty[f], 1);
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
  else consumer<EBT, EBD, PROBS>(P, sm, dyn, st);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&P.hdr->exit_cnt, 1u);
    if (d + 1u == gridDim.x) {
      P.hdr->ticket = 0u;
      P.hdr->exit_cnt = 0u;
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
  const uint32_t state = ld_relaxed(&pair_st(st, P.B, pair)->state);
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
