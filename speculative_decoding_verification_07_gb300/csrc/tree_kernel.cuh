// Token-tree verification: one cluster walks one request's tree at a time.
//
// Sources: "Keep cache validity aligned with the committed token history"
// (paragraph 3: a tree implementation keeps the accepted path; paragraph 5:
// test tree branch switches) and, for the law of each test, "Speculative
// decoding: accelerate LLM generation without changing its answers" sections
// 2-3.  At node j with children c_1 .. c_m (ascending node order) the children
// are tested in turn against the running residual of p_j:
//   p_1 = p_j,  p_{r+1} = normalize(max(0, p_r - q_j)),
// the first accepted child becomes the current node, the correction after m
// rejections is drawn from p_{m+1}, and a node without children gets the bonus
// from p_j.  The residuals are kept in closed form: p_r = max(0, p - c_r q)/W_r
// with c_1 = 0, W_1 = 1, c_{r+1} = c_r + W_r and W_{r+1} = sum max(0, p -
// c_{r+1} q), so a rejection costs one cluster-wide sum over the resident
// slices and no rewrite of them.
//
// The rows of the current node stay in the cluster's shared memory (one TMA
// bulk copy per row slice); the statistics, the top-k / top-p filters and the
// exponential race are the linear kernel's.  Requests are independent: the
// clusters take them from a ticket counter (walks differ in length, so a
// cluster that finishes early takes the next request) and never wait on one
// another.
#pragma once

#include "verify_kernel.cuh"

namespace sv {

struct TreeParams {
  int B, N, V;
  const char* target;  // [B][N+1][t_ld]
  int64_t t_ld;
  const char* draft;   // [B][N+1][d_ld]
  int64_t d_ld;
  const int32_t* parent;  // [B][N]
  const int32_t* tokens;  // [B][N]
  const int32_t* n_nodes; // [B] or null (= N)
  const float* temperature;
  const float* top_p;
  const int32_t* top_k;
  const uint32_t* request_id;
  const int32_t* seq_len;
  uint32_t seed_lo, seed_hi;
  int32_t* accepted;
  int32_t* path;        // [B][N]
  int32_t* out_tokens;  // [B][N+1]
  int32_t* num_emitted;
  uint32_t* status;
  const int32_t* eos;      // [B] or null
  const int32_t* max_new;  // [B] or null
  const float* rep_penalty;   // [B] or null
  const int32_t* rep_tokens;  // [B][rep_ld]
  int rep_ld;
  int rep_draft;  // 1: draft rows are logits and take the penalty too
  int* err;
  uint32_t* ctr;  // [2] request ticket and done counters, zero between calls
  int slice, d_off;
};

// The first child of node `cur` with index >= from (0: none).  Every warp
// scans 32 nodes per step and gets the same answer.
__device__ __forceinline__ int tree_next_child(const int32_t* par, int cur, int from, int n) {
  const int lane = threadIdx.x & 31;
  for (int j0 = from; j0 <= n; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t m = __ballot_sync(0xffffffffu, j <= n && par[j - 1] == cur);
    if (m) return j0 + __ffs(m) - 1;
  }
  return 0;
}

// Cluster-wide sum of one value per thread, reduced in a fixed order (lanes,
// warps, ranks), so every CTA gets the same bits.  Consecutive calls alternate
// the slot: a slot is rewritten only after a later call's barrier, which every
// peer passes after its reads of the slot.
__device__ __forceinline__ float tree_cluster_sum(cg::cluster_group& cluster, Smem& sm, float v,
                                                  int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sm.scratch_f[warp][0] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f;
    for (int w = 0; w < kWarps; ++w) a += sm.scratch_f[w][0];
    sm.kz[slot] = a;
  }
  cluster.sync();
  float s = 0.0f;
  const int C = (int)cluster.num_blocks();
  for (int r = 0; r < C; ++r) s += cluster.map_shared_rank(&sm, r)->kz[slot];
  return s;
}

// Statistics of the current node's target row (and draft row when has_d):
// raw maxima, then weight sums relative to them, each reduced across the
// cluster in a fixed order.  With win_t / win_d (bf16 logit rows under
// top-p alone) the sums sweep also counts the first top-p window into
// sm.hist[0], its floor taken from a lower bound of S known after the maxima
// (as in the linear kernel).  Returns false when a row is unusable.
template <int EBT, int EBD, bool PROBS>
__device__ bool tree_node_stats(cg::cluster_group& cluster, Smem& sm, const char* s_t,
                                const char* s_d, const SliceIter& it, bool has_d, float T,
                                float top_p, bool win_t, bool win_d, bool landed, RowP& rt,
                                RowP& rd) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = (int)cluster.num_blocks();
  const bool greedy = T == 0.0f;
  rt.greedy = rd.greedy = greedy;
  rt.c = greedy ? 0.0f : kLog2e / T;
  rt.invT = rd.invT = greedy ? 0.0f : 1.0f / T;
  rd.c = PROBS ? 1.0f : rt.c;
  rt.Dstar = rd.Dstar = kNoFilter;

  uint32_t mt2 = 0xFF80FF80u, md2 = 0xFF80FF80u;
  float rmt = -INFINITY, rmd = PROBS ? 0.0f : -INFINITY;
  for (int blk = 0; blk < it.nblk; ++blk) {
    const int x = it.x(blk);
    if (x < it.x1) {
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
  const float md = (PROBS && !greedy) ? (rmd > 0.0f ? lg2(rmd) * rd.invT : -INFINITY) : rmd;
  if (win_t || win_d)
    for (int j = threadIdx.x; j < 512; j += kThreads) (&sm.hist[0][0][0])[j] = 0u;
  {
    // every thread's own maximum weighs 1 relative to itself: the sum over
    // threads of 2^((m_thread - M) c) is a lower bound of S
    float Mt = rmt, Lt = rmt == -INFINITY ? 0.0f : 1.0f;
    float Md = md, Ld = md == -INFINITY ? 0.0f : 1.0f;
    warp_ms(Mt, Lt, rt.c, greedy);
    warp_ms(Md, Ld, rd.c, greedy);
    float Rm = rmd;
#pragma unroll
    for (int o = 16; o; o >>= 1) Rm = fmaxf(Rm, __shfl_xor_sync(0xffffffffu, Rm, o));
    const bool warp_bad = __any_sync(0xffffffffu, !landed);
    if (lane == 0)
      sm.part[warp] = {make_float4(Mt, Lt, Rm, warp_bad ? 1.0f : 0.0f), make_float4(Md, Ld, 0.0f, 0.0f)};
  }
  __syncthreads();
  if (warp == 0) {
    const StatPart c = combine_parts(lane < kWarps ? sm.part[lane] : neutral_part<PROBS>(), rt.c,
                                     rd.c, greedy);
    if (lane == 0) sm.cpart = c;
  }
  cluster.sync();
  bool slice_bad;
  float St_lb, Sd_lb;
  {
    const StatPart c = combine_parts(
        lane < C ? cluster.map_shared_rank(&sm, lane)->cpart : neutral_part<PROBS>(), rt.c, rd.c, greedy);
    rt.m = rt.mz = c.a.x;
    rd.m = c.a.z;
    rd.mz = c.d.x;
    St_lb = c.a.y, Sd_lb = c.d.y;
    slice_bad = c.a.w != 0.0f;
  }
  rt.kmax = vkey<EBT>(rt.m);
  rd.kmax = vkey<EBD>(rd.m);
  uint32_t thr2_t = 0x7FFF7FFFu, thr2_d = 0x7FFF7FFFu;  // NaN pairs: nothing passes
  const int nguess = min(it.V, kWindowGuess);
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

  float st = 0.0f, sd = 0.0f;
  uint32_t wt_lo = 0u, wt_hi = 0u, wd_lo = 0u, wd_hi = 0u;
  int wt_n = 0, wd_n = 0;
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
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    st += __shfl_xor_sync(0xffffffffu, st, o);
    sd += __shfl_xor_sync(0xffffffffu, sd, o);
  }
  if (lane == 0) sm.spart[warp] = make_float2(st, sd);
  __syncthreads();
  if (warp == 0) {
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
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
      v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    rt.S = v.x, rd.S = v.y;
    if (slice_bad) rt.S = __int_as_float(0x7FC00000);
  }
  rt.Z = rt.S, rd.Z = rd.S;
  rt.invZ = 1.0f / rt.Z, rd.invZ = 1.0f / rd.Z;
  rt.vstar = -INFINITY;
  rd.vstar = PROBS ? 0.0f : -INFINITY;
  const bool bad_t = !(rt.S >= 1.0f && rt.S <= FLT_MAX) || !(rt.m <= FLT_MAX) || rt.m == -INFINITY;
  const bool bad_d = has_d && (!(rd.S >= 1.0f && rd.S <= FLT_MAX) || !(rd.m <= FLT_MAX) ||
                               (PROBS ? !(rd.m > 0.0f) : rd.m == -INFINITY));
  return !bad_t && !bad_d;
}

// sum over this thread's slice elements of max(0, p(x) - c q(x)), with c
// folded into rdc.invZ
template <int EBT, int EBD, bool PROBS>
__device__ __forceinline__ float tree_residual_part(const char* s_t, const char* s_d,
                                                    const SliceIter& it, const RowP& rt,
                                                    const RowP& rdc) {
  float w = 0.0f;
  for (int blk = 0; blk < it.nblk; ++blk) {
    const int x = it.x(blk);
    if (x < it.x1) {
      Grp<EBT> g;
      Grp<EBD> h;
      lds_group<EBT, false>(g, s_t, it.x0, x, it.x1);
      lds_group<EBD, PROBS>(h, s_d, it.x0, x, it.x1);
#pragma unroll
      for (int e = 0; e < kGroup; ++e)
        w += fmaxf(0.0f, prob<EBT, false>(gval<EBT>(g, e), rt) - prob<EBD, PROBS>(gval<EBD>(h, e), rdc));
    }
  }
  return w;
}

template <int EB>
__device__ __forceinline__ float row_value(const char* row, int y) {
  return EB == 2 ? __uint_as_float((uint32_t)((const uint16_t*)row)[y] << 16) : ((const float*)row)[y];
}

// OPTS: the request options (EOS ids, output caps, repetition penalty) are
// compiled in; the plain variants leave their code out of the walk.
template <int EBT, int EBD, bool PROBS, bool OPTS>
__global__ void __launch_bounds__(kThreads, 2) tree_kernel(const TreeParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ Smem sm;
  __shared__ int s_ticket;
  extern __shared__ __align__(128) char dyn[];
  char* s_t = dyn;
  char* s_d = dyn + P.d_off;
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const bool lead = rank == 0 && tid == 0;
  const uint32_t k0 = P.seed_lo, k1 = P.seed_hi;
  uint32_t phase_t = 0u, phase_d = 0u;

  if (tid == 0) {
    mbar_init(&sm.bar[0]), mbar_init(&sm.bar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  SliceIter it;
  it.x0 = rank * P.slice;
  it.x1 = min(P.V, it.x0 + P.slice);
  it.nblk = it.x1 > it.x0 ? (it.x1 - it.x0 + kBlk - 1) / kBlk : 0;
  it.V = P.V;
  it.stride = kBlk, it.tid = (int)threadIdx.x;

  for (;;) {
    if (lead) s_ticket = (int)atomicAdd(P.ctr, 1u);
    cluster.sync();  // also: the previous request's shared memory is no longer read
    const int b = *cluster.map_shared_rank(&s_ticket, 0);
    cluster.sync();  // every CTA holds b before rank 0 takes the next ticket
    if (b >= P.B) break;
    const int N = P.N;
    const int n = P.n_nodes ? P.n_nodes[b] : N;
    const float T = P.temperature[b];
    const float top_p = P.top_p ? P.top_p[b] : 1.0f;
    const int top_k = P.top_k ? P.top_k[b] : 0;
    const uint32_t rid = P.request_id ? P.request_id[b] : (uint32_t)b;
    const int S = P.seq_len ? P.seq_len[b] : 0;
    const int eos = OPTS && P.eos ? P.eos[b] : -1;
    const int cap = OPTS && P.max_new ? P.max_new[b] : 0x7FFFFFFF;
    const float theta = OPTS && P.rep_penalty ? P.rep_penalty[b] : 1.0f;
    const bool rep = OPTS && theta != 1.0f;
    const int32_t* hist = P.rep_tokens + (size_t)b * P.rep_ld;
    const int32_t* par = P.parent + (size_t)b * N;
    const int32_t* tok = P.tokens + (size_t)b * N;
    int32_t* o_path = P.path + (size_t)b * N;
    int32_t* o_tok = P.out_tokens + (size_t)b * (N + 1);

    // the tree and the parameters are checked before any row is read
    bool bad = !(T >= 0.0f && T <= FLT_MAX) || !(top_p > 0.0f && top_p <= 1.0f) || n < 0 || n > N ||
               cap < 1 || !theta_valid(theta);
    if (!bad)
      for (int j = tid + 1; j <= n; j += kThreads) {
        const int pj = par[j - 1], yj = tok[j - 1];
        bad |= !(pj >= 0 && pj < j) || !(yj >= 0 && yj < P.V);
      }
    bad = __syncthreads_or(bad);

    // A node's rows head for shared memory as soon as the node is known (at
    // the request's start, or when its parent's test accepts it): every read
    // of the slices by this CTA lies before a barrier thread 0 has passed.
    auto issue = [&](int node) -> int {  // returns the node's first child (0: none)
      const int fc = tree_next_child(par, node, node + 1, n);
      if (tid == 0 && it.nblk > 0) {
        const char* tr = P.target + ((size_t)b * (N + 1) + node) * P.t_ld * EBT;
        const char* dr = P.draft + ((size_t)b * (N + 1) + node) * P.d_ld * EBD;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t bt = (uint32_t)(((it.x1 - it.x0) * EBT + 15) & ~15);
        mbar_expect_tx(&sm.bar[0], bt);
        bulk_g2s(s_t, tr + (size_t)it.x0 * EBT, bt, &sm.bar[0]);
        if (fc) {
          const uint32_t bd = (uint32_t)(((it.x1 - it.x0) * EBD + 15) & ~15);
          mbar_expect_tx(&sm.bar[1], bd);
          bulk_g2s(s_d, dr + (size_t)it.x0 * EBD, bd, &sm.bar[1]);
        }
      }
      return fc;
    };

    int cur = 0, depth = 0;
    uint32_t st_bits = 0u;
    int emitted = -1;  // the correction or bonus token, once drawn
    uint32_t stop = 0u;  // SV_ST_EOS / SV_ST_CAPPED: the walk ended on an accepted child
    int first = bad ? 0 : issue(0);
    while (!bad && emitted < 0 && !stop) {
      cluster.sync();  // the previous node's shared memory is no longer read anywhere
      const bool has_d = first > 0;
      const char* trow = P.target + ((size_t)b * (N + 1) + cur) * P.t_ld * EBT;
      const char* drow = P.draft + ((size_t)b * (N + 1) + cur) * P.d_ld * EBD;
      // repetition penalty: this node's set is the history plus the tokens of
      // the accepted path up to and including cur; its ids inside this slice
      // are marked in a bitmap while the rows load (each id once)
      uint32_t* rmask = reinterpret_cast<uint32_t*>(&sm.wb);
      const bool pen = rep && it.nblk > 0;
      if (pen) {
        for (int j = tid; j < kMaxBlk * kBlk / 32; j += kThreads) rmask[j] = 0u;
        __syncthreads();
        auto mark = [&](int x) {
          if (x >= it.x0 && x < it.x1) atomicOr(&rmask[(x - it.x0) >> 5], 1u << ((x - it.x0) & 31));
        };
        for (int j = tid; j < P.rep_ld; j += kThreads) mark(hist[j]);
        if (tid == 0)
          for (int a = cur; a > 0; a = par[a - 1]) mark(tok[a - 1]);
      }
      bool landed = true;
      if (it.nblk > 0) {
        landed &= mbar_wait(&sm.bar[0], phase_t, P.err);
        if (has_d) landed &= mbar_wait(&sm.bar[1], phase_d, P.err);
        phase_t ^= 1u;
        if (has_d) phase_d ^= 1u;
      }
      if (pen) {
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
      RowP rt, rd;
      const bool greedy = T == 0.0f;
      const bool topk = !greedy && top_k > 0 && top_k < P.V;
      // bf16 logit rows under top-p alone count their first window in the sums sweep
      const bool topp = !greedy && !topk && top_p < 1.0f;
      const bool win_t = EBT == 2 && topp, win_d = EBD == 2 && !PROBS && topp && has_d;
      if (!tree_node_stats<EBT, EBD, PROBS>(cluster, sm, s_t, s_d, it, has_d, T, top_p, win_t, win_d,
                                            landed, rt, rd)) {
        bad = true;
        break;
      }
      if (topk || topp)
        filter_rows<EBT, EBD, PROBS>(cluster, sm, s_t, s_d, it, has_d, top_p, topk ? top_k : 0, rt,
                                     rd, win_t, win_d);
      const uint32_t pos = (uint32_t)(S + depth + 1);
      RacePart best = {0.0f, 1.0f, 0x7FFFFFFF};
      if (!has_d) {  // a leaf: the bonus from p
        race_slice<EBT, EBD, PROBS>(s_t, s_d, it, false, rt, rd, pos, rid, k0, k1, sm.wb.idx[warp], best);
        emitted = race_reduce(cluster, sm, best, 0).idx;
        break;
      }
      // the children in turn, against the running residual max(0, p - c q) / W
      float c = 0.0f, W = 1.0f;
      int j = first, r = 0, taken = 0;
      bool empty = false;
      while (j > 0) {
        const int y = tok[j - 1];
        float vt = row_value<EBT>(trow, y), vq = row_value<EBD>(drow, y);
        if (rep) {  // is y in this node's penalised set?
          bool hit = false;
          for (int h = tid; h < P.rep_ld; h += kThreads) hit |= hist[h] == y;
          if (tid == 0)
            for (int a = cur; a > 0; a = par[a - 1]) hit |= tok[a - 1] == y;
          if (__syncthreads_or(hit)) {
            vt = penalised<EBT>(vt, theta);
            if (P.rep_draft) vq = penalised<EBD>(vq, theta);
          }
        }
        const float p_y = prob<EBT, false>(vt, rt);
        const float q_y = prob<EBD, PROBS>(vq, rd);
        RowP rdc = rd;
        rdc.invZ = c * rd.invZ;
        const float pr_y = fmaxf(0.0f, p_y - prob<EBD, PROBS>(vq, rdc)) / W;
        const uint4 rr = philox4x32_10(make_uint4((uint32_t)r >> 2, pos, rid, 1u), k0, k1);
        const uint32_t sel = (r & 3) == 0 ? rr.x : (r & 3) == 1 ? rr.y : (r & 3) == 2 ? rr.z : rr.w;
        const float u = uniform_from_bits(sel);
        if (q_y == 0.0f) st_bits |= SV_ST_Q_ZERO;
        if (u * q_y < pr_y) {
          taken = j;
          break;
        }
        c += W;
        const int jn = tree_next_child(par, cur, j + 1, n);
        if (!jn) break;  // the last child: the correction needs c, not the new W
        rdc.invZ = c * rd.invZ;
        W = tree_cluster_sum(cluster, sm, tree_residual_part<EBT, EBD, PROBS>(s_t, s_d, it, rt, rdc),
                             r & 1);
        if (!(W > 0.0f)) {
          empty = true;
          break;
        }
        j = jn;
        ++r;
      }
      if (taken) {
        if (lead) o_path[depth] = taken, o_tok[depth] = tok[taken - 1];
        cur = taken;
        ++depth;
        // an accepted EOS id, or the cap's last token, ends the walk here
        if constexpr (OPTS) {
          if (eos >= 0 && tok[taken - 1] == eos) stop = SV_ST_EOS;
          else if (depth == cap) stop = SV_ST_CAPPED;
          if (stop) break;
        }
        first = issue(cur);
        continue;
      }
      // every child rejected: the correction from the last residual (from p
      // when that residual is numerically empty: found while testing, or as a
      // race whose winner weighs nothing)
      RowP rdc = rd;
      rdc.invZ = c * rd.invZ;
      RacePart win = {0.0f, 1.0f, 0x7FFFFFFF};
      if (!empty) {
        race_slice<EBT, EBD, PROBS>(s_t, s_d, it, true, rt, rdc, pos, rid, k0, k1, sm.wb.idx[warp], best);
        win = race_reduce(cluster, sm, best, 0);
        empty = !(win.w > 0.0f);
      }
      if (empty) {
        st_bits |= SV_ST_RESIDUAL_EMPTY;
        best = {0.0f, 1.0f, 0x7FFFFFFF};
        race_slice<EBT, EBD, PROBS>(s_t, s_d, it, false, rt, rd, pos, rid, k0, k1, sm.wb.idx[warp], best);
        win = race_reduce(cluster, sm, best, 1);
      }
      emitted = win.idx;
    }
    if (lead) {
      if (bad) {
        P.accepted[b] = -1;
        P.num_emitted[b] = 0;
        P.status[b] = SV_ST_BAD_INPUT;
        for (int q = 0; q < N; ++q) o_path[q] = -1;
        for (int q = 0; q <= N; ++q) o_tok[q] = -1;
      } else {
        const int ne = stop ? depth : depth + 1;
        if (!stop) o_tok[depth] = emitted;
        for (int q = depth; q < N; ++q) o_path[q] = -1;
        for (int q = ne; q <= N; ++q) o_tok[q] = -1;
        P.accepted[b] = depth;
        P.num_emitted[b] = ne;
        P.status[b] = st_bits | stop;
      }
    }
  }
  // the last cluster to finish resets the counters for the next call
  if (lead) {
    __threadfence();
    const uint32_t nclusters = gridDim.x / (uint32_t)C;
    if (atomicAdd(P.ctr + 1, 1u) == nclusters - 1) {
      P.ctr[0] = 0u;
      P.ctr[1] = 0u;
      __threadfence();
    }
  }
  cluster.sync();  // peers are done reading this CTA's shared memory
}

using TreeKernelFn = void (*)(TreeParams);
TreeKernelFn tree_kernel_bf16_bf16_logits();
TreeKernelFn tree_kernel_bf16_f32_probs();
TreeKernelFn tree_kernel_bf16_f32_logits();
TreeKernelFn tree_kernel_f32_f32_logits();
TreeKernelFn tree_kernel_f32_f32_probs();
TreeKernelFn tree_kernel_f32_bf16_logits();
TreeKernelFn tree_kernel_bf16_bf16_logits_opts();
TreeKernelFn tree_kernel_bf16_f32_probs_opts();
TreeKernelFn tree_kernel_bf16_f32_logits_opts();
TreeKernelFn tree_kernel_f32_f32_logits_opts();
TreeKernelFn tree_kernel_f32_f32_probs_opts();
TreeKernelFn tree_kernel_f32_bf16_logits_opts();

}  // namespace sv
