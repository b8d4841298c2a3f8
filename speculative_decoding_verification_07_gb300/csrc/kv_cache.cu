// Paged-KV bookkeeping around the verification step: block free list,
// lookahead reserve, commit / rollback, prefix fork, release, and the
// contiguous write-pointer rollback.
//
// Sources: "Walk through KV-cache updates when speculative decoding rejects
// some draft tokens" (free the pages covering rejected positions / rewind the
// write pointer; the cache then holds exactly the committed sequence);
// "Rejected speculative tokens remain in KV", paragraphs 1-2 (allocation is not
// acceptance; a block may stay with only part of it valid); "Keep cache
// validity aligned with the committed token history", paragraphs 1-4 (pending
// token, block tables / ownership / reference counts, shared-prefix isolation).
//
// Every kernel here touches kilobytes of metadata, so each runs as ONE block of
// 1024 threads: requests are spread over threads, block-wide scans fix the
// (request, block) order of every pop and push, and validation runs before any
// mutation so that a refused call leaves the pool unchanged.  K/V payload is
// never read or written.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace sv {

constexpr int kKvThreads = 1024;

// Threads of the one-block kernels: one per item up to 1024, whole warps.
// Fewer idle warps make every block barrier and scan cheaper.
static int kv_threads(int n) {
  const int t = ((n > 0 ? n : 1) + 31) / 32 * 32;
  return t < kKvThreads ? t : kKvThreads;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Exclusive block-wide scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total.
__device__ int block_excl_scan(int v, int* scratch /*[32]*/, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    scratch[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int off = warp ? scratch[warp - 1] : 0;
  const int tot = scratch[(blockDim.x >> 5) - 1];
  __syncthreads();
  *total = tot;
  return off + x - v;
}

__global__ void bfl_init_kernel(bfl_state st) {
  const int n = st.num_blocks;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    st.free_stack[i] = n - 1 - i;
    st.refcount[i] = 0;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *st.free_top = n;
}

// ---------------------------------------------------------------------------
// Lookahead reserve: cover [0, S_b + k_b + 1) for every request, all or nothing.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kKvThreads) bfl_reserve_kernel(bfl_state st, int B,
                                                                 const int32_t* seq_len,
                                                                 const int32_t* k, int32_t* table,
                                                                 int max_blocks, int* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int scratch[32];
  __shared__ int s_err;
  const int BS = st.block_size, nb = st.num_blocks;
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  int total = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int need = 0;
    if (b < B) {
      const int S = seq_len[b], kb = k ? k[b] : 0;
      const int have = ceil_div(S, BS), want = ceil_div(S + kb + 1, BS);
      const int32_t* row = table + (size_t)b * max_blocks;
      bool bad = S < 0 || kb < 0 || want > max_blocks;
      if (!bad && have > 0) {
        const int last = row[have - 1];
        bad = last < 0 || last >= nb;
        // appending into a partially filled block that is shared is refused
        if (!bad && (S % BS) != 0 && st.refcount[last] > 1) bad = true;
      }
      for (int j = have; !bad && j < want; ++j) bad = row[j] >= 0;
      if (bad) atomicExch(&s_err, 1);
      need = bad ? 0 : want - have;
    }
    int t;
    block_excl_scan(need, scratch, &t);
    total += t;
  }
  __syncthreads();
  const int top = *st.free_top;
  if (s_err) {
    if (threadIdx.x == 0) report(err, SV_ERR_STATE);
    return;
  }
  if (total > top) {
    if (threadIdx.x == 0) report(err, SV_ERR_OOM);
    return;
  }
  int running = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int need = 0, have = 0;
    if (b < B) {
      const int S = seq_len[b], kb = k ? k[b] : 0;
      have = ceil_div(S, BS);
      need = ceil_div(S + kb + 1, BS) - have;
    }
    int t;
    const int excl = block_excl_scan(need, scratch, &t) + running;
    if (b < B) {
      int32_t* row = table + (size_t)b * max_blocks;
      for (int j = 0; j < need; ++j) {
        const int blk = st.free_stack[top - 1 - (excl + j)];
        row[have + j] = blk;
        st.refcount[blk] = 1;
      }
    }
    running += t;
  }
  __syncthreads();
  if (threadIdx.x == 0) *st.free_top = top - total;
}

// ---------------------------------------------------------------------------
// Shared machinery for dropping blocks in a fixed (item, j) order.
//
// Each item (a request) drops the table entries j in [j0, j1) of one row.
// Sequential semantics: walking items ascending and j ascending, decrement the
// refcount and push the block when it reaches 0.  In parallel: decrement with
// atomics; if every decrement saw 1 (no block dropped twice, none shared) each
// drop is its block's only dropper and pushes.  Otherwise the LAST dropper in
// walk order of each block that reached 0 is found by an atomicMin of
// -(1 + walk index) into the (now zero) refcount, then the refcount is reset.
// Pushes are placed by a block-wide scan in walk order.
// ---------------------------------------------------------------------------
struct DropRange {
  int32_t* row;
  int j0, j1;
};

template <class RangeFn, class DoneFn>
__device__ bool drop_blocks(const bfl_state& st, int n_items, int max_blocks, RangeFn range,
                            DoneFn done, int* err) {
  __shared__ int scratch[32];
  __shared__ int s_err;
  const int nb = st.num_blocks;
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  // 1. validate every drop before mutating anything
  for (int base = 0; base < n_items; base += blockDim.x) {
    const int it = base + threadIdx.x;
    if (it < n_items) {
      DropRange r = range(it);
      if (r.j0 < 0) atomicExch(&s_err, 1);
      for (int j = max(r.j0, 0); j < r.j1; ++j) {
        const int blk = r.row[j];
        if (blk < 0 || blk >= nb || st.refcount[blk] <= 0) atomicExch(&s_err, 1);
      }
    }
  }
  __syncthreads();
  if (s_err) {
    if (threadIdx.x == 0) report(err, SV_ERR_STATE);
    return false;
  }
  // 2. decrement
  int shared_seen = 0;
  for (int base = 0; base < n_items; base += blockDim.x) {
    const int it = base + threadIdx.x;
    if (it < n_items) {
      DropRange r = range(it);
      for (int j = r.j0; j < r.j1; ++j)
        shared_seen |= atomicSub(&st.refcount[r.row[j]], 1) != 1;
    }
  }
  const bool slow = __syncthreads_or(shared_seen);
  // 3. slow path: mark the last dropper of every block that reached zero
  if (slow) {
    for (int base = 0; base < n_items; base += blockDim.x) {
      const int it = base + threadIdx.x;
      if (it < n_items) {
        DropRange r = range(it);
        for (int j = r.j0; j < r.j1; ++j) {
          const int blk = r.row[j];
          if (st.refcount[blk] <= 0) atomicMin(&st.refcount[blk], -(1 + it * max_blocks + j));
        }
      }
    }
    __syncthreads();
  }
  // 4. count pushes per item, scan, push, clear table entries
  const int top = *st.free_top;
  int running = 0;
  for (int base = 0; base < n_items; base += blockDim.x) {
    const int it = base + threadIdx.x;
    DropRange r{nullptr, 0, 0};
    int pushes = 0;
    if (it < n_items) {
      r = range(it);
      if (!slow) {
        pushes = r.j1 - r.j0;
      } else {
        for (int j = r.j0; j < r.j1; ++j)
          pushes += st.refcount[r.row[j]] == -(1 + it * max_blocks + j);
      }
    }
    int t;
    const int excl = block_excl_scan(pushes, scratch, &t) + running;
    if (it < n_items) {
      int p = 0;
      for (int j = r.j0; j < r.j1; ++j) {
        const int blk = r.row[j];
        if (!slow || st.refcount[blk] == -(1 + it * max_blocks + j))
          st.free_stack[top + excl + p++] = blk;
      }
      done(it, pushes);
    }
    running += t;
  }
  __syncthreads();
  if (slow) {  // every marked block goes back to refcount 0; then clear the rows
    for (int base = 0; base < n_items; base += blockDim.x) {
      const int it = base + threadIdx.x;
      if (it < n_items) {
        DropRange r = range(it);
        for (int j = r.j0; j < r.j1; ++j)
          if (st.refcount[r.row[j]] < 0) st.refcount[r.row[j]] = 0;
      }
    }
    __syncthreads();
  }
  for (int base = 0; base < n_items; base += blockDim.x) {
    const int it = base + threadIdx.x;
    if (it < n_items) {
      DropRange r = range(it);
      for (int j = r.j0; j < r.j1; ++j) r.row[j] = -1;
    }
  }
  if (threadIdx.x == 0) *st.free_top = top + running;
  return true;
}

// ---------------------------------------------------------------------------
// Commit / rollback after the verify pass.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kKvThreads) kv_commit_kernel(bfl_state st, int B,
                                                               const int32_t* k,
                                                               const int32_t* accepted,
                                                               int32_t* seq_len, int32_t* table,
                                                               int max_blocks, int32_t* n_freed,
                                                               int* err) {
  pdl_wait();
  pdl_trigger();
  const int BS = st.block_size;
  // accepted outside [-1, k_b] or a held range beyond the table: refuse the call
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int S = seq_len[b], kb = k ? k[b] : 0, a = accepted[b];
    if (S < 0 || kb < 0 || a < -1 || a > kb || ceil_div(S + kb + 1, BS) > max_blocks)
      atomicExch(&s_bad, 1);
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) report(err, SV_ERR_STATE);
    return;
  }
  auto range = [&](int b) {
    const int S = seq_len[b], kb = k ? k[b] : 0, a = accepted[b];
    const int nw = a < 0 ? S : S + 1 + a;
    return DropRange{table + (size_t)b * max_blocks, ceil_div(nw, BS), ceil_div(S + kb + 1, BS)};
  };
  auto done = [&](int b, int pushes) {
    if (n_freed) n_freed[b] = pushes;
  };
  const bool ok = drop_blocks(st, B, max_blocks, range, done, err);
  __syncthreads();  // range() reads seq_len: update it only after every drop
  if (!ok) return;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int S = seq_len[b], a = accepted[b];
    seq_len[b] = a < 0 ? S : S + 1 + a;
  }
}

// ---------------------------------------------------------------------------
// Lookahead reserve with copy-on-write of a shared partial last block.
// Bookkeeping (one block): pops in (request, j) order with the copy first, the
// copy list to cow[b] = (old, new, r), then the old blocks dropped in request
// order and the copies installed.  kv_cow_copy_kernel moves the payload.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kKvThreads) bfl_reserve_cow_kernel(bfl_state st, int B,
                                                                     const int32_t* seq_len,
                                                                     const int32_t* k, int32_t* table,
                                                                     int max_blocks, int32_t* cow,
                                                                     int* err) {
  __shared__ int scratch[32];
  __shared__ int s_err;
  const int BS = st.block_size, nb = st.num_blocks;
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  int total = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int need = 0;
    if (b < B) {
      const int S = seq_len[b], kb = k ? k[b] : 0;
      const int have = ceil_div(S, BS), want = ceil_div(S + kb + 1, BS);
      const int32_t* row = table + (size_t)b * max_blocks;
      bool bad = S < 0 || kb < 0 || want > max_blocks;
      for (int j = 0; !bad && j < have; ++j) bad = row[j] < 0 || row[j] >= nb;
      for (int j = have; !bad && j < want; ++j) bad = row[j] >= 0;
      if (bad) atomicExch(&s_err, 1);
      const bool c = !bad && (S % BS) != 0 && st.refcount[row[have - 1]] > 1;
      need = bad ? 0 : want - have + (c ? 1 : 0);
      cow[3 * b] = c ? row[have - 1] : -1;
      cow[3 * b + 1] = -1;
      cow[3 * b + 2] = c ? S % BS : 0;
    }
    int t;
    block_excl_scan(need, scratch, &t);
    total += t;
  }
  __syncthreads();
  const int top = *st.free_top;
  if (s_err || total > top) {  // refused: no copy may run either
    for (int b = threadIdx.x; b < B; b += blockDim.x) cow[3 * b] = -1;
    if (threadIdx.x == 0) report(err, s_err ? SV_ERR_STATE : SV_ERR_OOM);
    return;
  }
  int running = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int need = 0, have = 0, c = 0;
    if (b < B) {
      const int S = seq_len[b], kb = k ? k[b] : 0;
      have = ceil_div(S, BS);
      c = cow[3 * b] >= 0 ? 1 : 0;
      need = ceil_div(S + kb + 1, BS) - have + c;
    }
    int t;
    const int excl = block_excl_scan(need, scratch, &t) + running;
    if (b < B) {
      int32_t* row = table + (size_t)b * max_blocks;
      for (int j = 0; j < need; ++j) {
        const int blk = st.free_stack[top - 1 - (excl + j)];
        st.refcount[blk] = 1;
        if (c && j == 0) cow[3 * b + 1] = blk;  // the copy: installed after the drops
        else row[have + j - c] = blk;
      }
      if (!c) cow[3 * b + 1] = -1;
    }
    running += t;
  }
  __syncthreads();
  if (threadIdx.x == 0) *st.free_top = top - total;
  __syncthreads();
  // the shared blocks lose one reference per copy (pushed if none is left)
  auto range = [&](int b) {
    const int S = seq_len[b];
    const int have = ceil_div(S, BS);
    return cow[3 * b] >= 0 ? DropRange{table + (size_t)b * max_blocks, have - 1, have}
                           : DropRange{table + (size_t)b * max_blocks, 0, 0};
  };
  auto done = [&](int, int) {};
  drop_blocks(st, B, max_blocks, range, done, err);
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x)
    if (cow[3 * b] >= 0) table[(size_t)b * max_blocks + ceil_div(seq_len[b], BS) - 1] = cow[3 * b + 1];
}

// Payload of the copy-on-write blocks: slots [0, r) of every (layer, K/V,
// head) run, old -> new.  Grid: B x kCowSplit CTAs, 16-byte vectors.
constexpr int kCowSplit = 8;

__global__ void kv_cow_copy_kernel(int B, const int32_t* cow, kv_payload kv, int block_size) {
  const int b = blockIdx.x / kCowSplit, part = blockIdx.x % kCowSplit;
  if (b >= B) return;
  const int old = cow[3 * b], nw = cow[3 * b + 1], r = cow[3 * b + 2];
  if (old < 0 || nw < 0 || r <= 0) return;
  const int runs = kv.layers * 2 * kv.heads;
  const size_t run = (size_t)block_size * kv.head_dim * kv.elem_bytes;  // bytes of one (l, kv, h) run
  const int vec = (int)((size_t)r * kv.head_dim * kv.elem_bytes / 16);  // 16-byte vectors to copy per run
  const char* src = static_cast<const char*>(kv.data) + (size_t)old * runs * run;
  char* dst = static_cast<char*>(kv.data) + (size_t)nw * runs * run;
  for (int q = part; q < runs; q += kCowSplit) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)q * run);
    uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)q * run);
    for (int v = threadIdx.x; v < vec; v += blockDim.x) d4[v] = s4[v];
  }
}

// ---------------------------------------------------------------------------
// Commit by copy: staged K/V of positions S_b .. S_b + a_b into paged slots.
// kCopySplit CTAs per (request, entry) share its layers x 2 x heads runs of
// head_dim elements; every thread keeps 4 16-byte loads in flight.  The
// register cap (32 a thread, eight CTAs per SM) is what makes the paged
// destination as fast as a contiguous one: at 74 registers only three CTAs fit
// on an SM, most of the grid waits for a slot, and the copy took 30 % longer.
// ---------------------------------------------------------------------------
constexpr int kCopySplit = 8;

// rows: positions S_b .. S_b + rows - 1 considered per request; entries: the
// stage's entries per request; path (tree commits) [B][path_ld]: the entry of
// position S_b + i is path[b][i - 1] for i >= 1 (NULL: entry i).
__global__ void __launch_bounds__(256, 8) kv_commit_copy_kernel(int B, int rows, int entries,
                                                             const int32_t* path, int path_ld,
                                                             const int32_t* accepted,
                                                             const int32_t* seq_len,
                                                             const int32_t* table, int max_blocks,
                                                             int block_size, int num_blocks,
                                                             const char* stage, kv_payload kv,
                                                             int* err) {
  const int e = blockIdx.x / kCopySplit, part = blockIdx.x % kCopySplit;
  const int b = e / rows, i = e % rows;
  if (b >= B) return;
  const int a = accepted[b];
  if (i == 0 && part == 0 && a >= rows && threadIdx.x == 0) report(err, SV_ERR_STATE);  // path too long
  if (i > a) return;
  int src_entry = i;
  if (path && i > 0) {
    src_entry = path[(size_t)b * path_ld + i - 1];
    if (src_entry < 1 || src_entry >= entries) {
      if (threadIdx.x == 0 && part == 0) report(err, SV_ERR_STATE);
      return;
    }
  }
  const int p = seq_len[b] + i;
  const int j = p / block_size;
  const int blk = (p >= 0 && j < max_blocks) ? table[(size_t)b * max_blocks + j] : -1;
  if (blk < 0 || blk >= num_blocks) {
    if (threadIdx.x == 0 && part == 0) report(err, SV_ERR_STATE);
    return;
  }
  const int runs = kv.layers * 2 * kv.heads;
  const int vrun = kv.head_dim * kv.elem_bytes / 16;  // 16-byte vectors per run
  const size_t run = (size_t)block_size * kv.head_dim * kv.elem_bytes;
  const uint4* src = reinterpret_cast<const uint4*>(
      stage + ((size_t)b * entries + src_entry) * runs * kv.head_dim * kv.elem_bytes);
  char* dst = static_cast<char*>(kv.data) + (size_t)blk * runs * run +
              (size_t)(p % block_size) * kv.head_dim * kv.elem_bytes;
  const int n = runs * vrun;
  const int v0 = (int)((long long)n * part / kCopySplit), v1 = (int)((long long)n * (part + 1) / kCopySplit);
  constexpr int kU = 4;
  for (int base = v0 + threadIdx.x; base < v1; base += kU * blockDim.x) {
    uint4 r[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * blockDim.x;
      if (v < v1) r[u] = src[v];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * blockDim.x;
      if (v < v1) {
        const int q = v / vrun, w = v - q * vrun;
        reinterpret_cast<uint4*>(dst + (size_t)q * run)[w] = r[u];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Draft-cache realignment: the draft keeps min(D_b, committed length) of its
// own processed positions and drops the blocks past them.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kKvThreads) kv_commit_draft_kernel(bfl_state st, int B,
                                                                     const int32_t* seq_len,
                                                                     const int32_t* accepted,
                                                                     int32_t* draft_len,
                                                                     int32_t* table, int max_blocks,
                                                                     int32_t* n_freed, int* err) {
  const int BS = st.block_size, nb = st.num_blocks;
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int S = seq_len[b], a = accepted[b], D = draft_len[b];
    bool bad = S < 0 || D < 0 || a < -1 || ceil_div(D, BS) > max_blocks;
    const int32_t* row = table + (size_t)b * max_blocks;
    for (int j = 0; !bad && j < ceil_div(D, BS); ++j) bad = row[j] < 0 || row[j] >= nb;
    if (bad) atomicExch(&s_bad, 1);
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) report(err, SV_ERR_STATE);
    return;
  }
  auto keep_of = [&](int b) {
    const int S = seq_len[b], a = accepted[b], D = draft_len[b];
    const int c = a < 0 ? S : S + 1 + a;
    return c < D ? c : D;
  };
  auto range = [&](int b) {
    return DropRange{table + (size_t)b * max_blocks, ceil_div(keep_of(b), BS),
                     ceil_div(draft_len[b], BS)};
  };
  auto done = [&](int b, int pushes) {
    if (n_freed) n_freed[b] = pushes;
  };
  const bool ok = drop_blocks(st, B, max_blocks, range, done, err);
  __syncthreads();  // range() reads draft_len: update it only after every drop
  if (!ok) return;
  for (int b = threadIdx.x; b < B; b += blockDim.x) draft_len[b] = keep_of(b);
}

// ---------------------------------------------------------------------------
// Release finished requests: drop every block they hold.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kKvThreads) bfl_release_kernel(bfl_state st, int n,
                                                                 const int32_t* req_ids,
                                                                 int32_t* seq_len, int32_t* table,
                                                                 int n_rows, int max_blocks,
                                                                 int32_t* n_freed, int* err) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int it = threadIdx.x; it < n; it += blockDim.x)
    if (req_ids[it] < 0 || req_ids[it] >= n_rows) atomicExch(&s_bad, 1);
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) report(err, SV_ERR_STATE);
    return;
  }
  auto range = [&](int it) {
    const int b = req_ids[it];
    int32_t* row = table + (size_t)b * max_blocks;
    int j1 = 0;
    while (j1 < max_blocks && row[j1] >= 0) ++j1;
    return DropRange{row, 0, j1};
  };
  auto done = [&](int it, int pushes) {
    if (n_freed) n_freed[it] = pushes;
  };
  const bool ok = drop_blocks(st, n, max_blocks, range, done, err);
  __syncthreads();
  if (!ok) return;
  for (int it = threadIdx.x; it < n; it += blockDim.x) seq_len[req_ids[it]] = 0;
}

// ---------------------------------------------------------------------------
// Fork: share whole blocks of src with dst (refcount + 1 each).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kKvThreads) bfl_fork_kernel(bfl_state st, int n_pairs,
                                                              const int32_t* src,
                                                              const int32_t* dst,
                                                              const int32_t* n_blocks,
                                                              int32_t* table, int n_rows,
                                                              int max_blocks, int* err) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int nb = st.num_blocks;
  for (int p = threadIdx.x; p < n_pairs; p += blockDim.x) {
    const int n = n_blocks[p];
    if (n < 0 || n > max_blocks || src[p] == dst[p] || src[p] < 0 || src[p] >= n_rows ||
        dst[p] < 0 || dst[p] >= n_rows) {
      atomicExch(&s_bad, 1);
      continue;
    }
    const int32_t* rs = table + (size_t)src[p] * max_blocks;
    const int32_t* rd = table + (size_t)dst[p] * max_blocks;
    for (int j = 0; j < n; ++j)
      if (rs[j] < 0 || rs[j] >= nb || rd[j] >= 0 || st.refcount[rs[j]] <= 0) atomicExch(&s_bad, 1);
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) report(err, SV_ERR_STATE);
    return;
  }
  for (int p = threadIdx.x; p < n_pairs; p += blockDim.x) {
    const int32_t* rs = table + (size_t)src[p] * max_blocks;
    int32_t* rd = table + (size_t)dst[p] * max_blocks;
    for (int j = 0; j < n_blocks[p]; ++j) {
      rd[j] = rs[j];
      atomicAdd(&st.refcount[rs[j]], 1);
    }
  }
}

__global__ void kv_rollback_contig_kernel(int B, const int32_t* accepted, int32_t* write_ptr) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int a = accepted[b];
    if (a >= 0) write_ptr[b] += 1 + a;
  }
}

static bool bad_state(const bfl_state* st) {
  return !st || st->num_blocks < 0 || st->block_size < 1 || !st->free_top ||
         (st->num_blocks > 0 && (!st->free_stack || !st->refcount));
}

}  // namespace sv

using namespace sv;

extern "C" sv_status bfl_init(sv_handle* h, const bfl_state* st, sv_stream_t stream) {
  if (!h || bad_state(st)) return SV_ERR_INVALID;
  const int grid = st->num_blocks > 0 ? (st->num_blocks + 255) / 256 : 1;
  bfl_init_kernel<<<grid < 4096 ? grid : 4096, 256, 0, (cudaStream_t)stream>>>(*st);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status bfl_reserve(sv_handle* h, const bfl_state* st, int32_t B,
                                 const int32_t* seq_len, const int32_t* k, int32_t* table,
                                 int32_t max_blocks, sv_stream_t stream) {
  if (!h || bad_state(st) || B < 0 || max_blocks < 1) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!seq_len || !table) return SV_ERR_INVALID;
  if (sv_launch_pdl(bfl_reserve_kernel, dim3(1), dim3(kv_threads(B)), 0, (cudaStream_t)stream, *st, B,
                    seq_len, k, table, (int)max_blocks, h->d_err) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

extern "C" sv_status bfl_fork_prefix(sv_handle* h, const bfl_state* st, int32_t n_pairs,
                                     const int32_t* src, const int32_t* dst,
                                     const int32_t* n_blocks, int32_t* table, int32_t n_rows,
                                     int32_t max_blocks, sv_stream_t stream) {
  if (!h || bad_state(st) || n_pairs < 0 || n_rows < 0 || max_blocks < 1) return SV_ERR_INVALID;
  if (n_pairs == 0) return SV_OK;
  if (!src || !dst || !n_blocks || !table) return SV_ERR_INVALID;
  bfl_fork_kernel<<<1, kv_threads(n_pairs), 0, (cudaStream_t)stream>>>(*st, n_pairs, src, dst, n_blocks,
                                                              table, n_rows, max_blocks, h->d_err);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status bfl_release(sv_handle* h, const bfl_state* st, int32_t n,
                                 const int32_t* req_ids, int32_t* seq_len, int32_t* table,
                                 int32_t n_rows, int32_t max_blocks, int32_t* n_freed,
                                 sv_stream_t stream) {
  if (!h || bad_state(st) || n < 0 || n_rows < 0 || max_blocks < 1) return SV_ERR_INVALID;
  if (n == 0) return SV_OK;
  if (!req_ids || !seq_len || !table) return SV_ERR_INVALID;
  bfl_release_kernel<<<1, kv_threads(n), 0, (cudaStream_t)stream>>>(*st, n, req_ids, seq_len, table,
                                                                 n_rows, max_blocks, n_freed,
                                                                 h->d_err);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status kv_commit_rollback(sv_handle* h, const bfl_state* st, int32_t B,
                                        const int32_t* k, const int32_t* accepted,
                                        int32_t* seq_len, int32_t* table, int32_t max_blocks,
                                        int32_t* n_freed, sv_stream_t stream) {
  if (!h || bad_state(st) || B < 0 || max_blocks < 1) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!accepted || !seq_len || !table) return SV_ERR_INVALID;
  if (sv_launch_pdl(kv_commit_kernel, dim3(1), dim3(kv_threads(B)), 0, (cudaStream_t)stream, *st, B, k,
                    accepted, seq_len, table, (int)max_blocks, n_freed, h->d_err) != cudaSuccess) {
    (void)cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

static bool bad_payload(const kv_payload* kv) {
  return !kv || !kv->data || ((uintptr_t)kv->data & 15u) || kv->layers < 1 || kv->heads < 1 ||
         kv->head_dim < 1 || (kv->elem_bytes != 2 && kv->elem_bytes != 4) ||
         ((size_t)kv->head_dim * kv->elem_bytes) % 16;
}

extern "C" sv_status bfl_reserve_cow(sv_handle* h, const bfl_state* st, int32_t B,
                                     const int32_t* seq_len, const int32_t* k, int32_t* table,
                                     int32_t max_blocks, const kv_payload* kv, int32_t* cow_scratch,
                                     sv_stream_t stream) {
  if (!h || bad_state(st) || B < 0 || max_blocks < 1 || bad_payload(kv)) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!seq_len || !table || !cow_scratch) return SV_ERR_INVALID;
  bfl_reserve_cow_kernel<<<1, kv_threads(B), 0, (cudaStream_t)stream>>>(*st, B, seq_len, k, table,
                                                                       max_blocks, cow_scratch,
                                                                       h->d_err);
  kv_cow_copy_kernel<<<B * kCowSplit, 256, 0, (cudaStream_t)stream>>>(B, cow_scratch, *kv,
                                                                      st->block_size);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status kv_commit_copy(sv_handle* h, int32_t B, int32_t kmax, const int32_t* accepted,
                                    const int32_t* seq_len, const int32_t* table, int32_t max_blocks,
                                    int32_t block_size, int32_t num_blocks, const void* stage,
                                    const kv_payload* kv, sv_stream_t stream) {
  if (!h || B < 0 || kmax < 0 || max_blocks < 1 || block_size < 1 || num_blocks < 0 ||
      bad_payload(kv) || ((uintptr_t)stage & 15u))
    return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!accepted || !seq_len || !table || !stage) return SV_ERR_INVALID;
  kv_commit_copy_kernel<<<B * (kmax + 1) * kCopySplit, 256, 0, (cudaStream_t)stream>>>(
      B, kmax + 1, kmax + 1, nullptr, 0, accepted, seq_len, table, max_blocks, block_size, num_blocks,
      static_cast<const char*>(stage), *kv, h->d_err);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status kv_commit_tree(sv_handle* h, int32_t B, int32_t N, int32_t max_depth,
                                    const int32_t* accepted, const int32_t* path,
                                    const int32_t* seq_len, const int32_t* table, int32_t max_blocks,
                                    int32_t block_size, int32_t num_blocks, const void* stage,
                                    const kv_payload* kv, sv_stream_t stream) {
  if (!h || B < 0 || N < 0 || max_depth < 0 || max_depth > N || max_blocks < 1 || block_size < 1 ||
      num_blocks < 0 || bad_payload(kv) || ((uintptr_t)stage & 15u))
    return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!accepted || !seq_len || !table || !stage || (N > 0 && !path)) return SV_ERR_INVALID;
  kv_commit_copy_kernel<<<B * (max_depth + 1) * kCopySplit, 256, 0, (cudaStream_t)stream>>>(
      B, max_depth + 1, N + 1, path, N, accepted, seq_len, table, max_blocks, block_size,
      num_blocks, static_cast<const char*>(stage), *kv, h->d_err);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status kv_commit_draft(sv_handle* h, const bfl_state* st, int32_t B,
                                     const int32_t* seq_len, const int32_t* accepted,
                                     int32_t* draft_len, int32_t* draft_table, int32_t max_blocks,
                                     int32_t* n_freed, sv_stream_t stream) {
  if (!h || bad_state(st) || B < 0 || max_blocks < 1) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!seq_len || !accepted || !draft_len || !draft_table) return SV_ERR_INVALID;
  kv_commit_draft_kernel<<<1, kv_threads(B), 0, (cudaStream_t)stream>>>(
      *st, B, seq_len, accepted, draft_len, draft_table, max_blocks, n_freed, h->d_err);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status kv_rollback_contig(sv_handle* h, int32_t B, const int32_t* accepted,
                                        int32_t* write_ptr, sv_stream_t stream) {
  if (!h || B < 0) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!accepted || !write_ptr) return SV_ERR_INVALID;
  kv_rollback_contig_kernel<<<(B + 255) / 256, 256, 0, (cudaStream_t)stream>>>(B, accepted,
                                                                               write_ptr);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
