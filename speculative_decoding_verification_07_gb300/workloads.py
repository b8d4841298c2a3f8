"""Seeded synthetic inputs for the batched verification step.

This module only synthesises inputs.  It holds none of the verifier's
arithmetic and imports neither the oracle nor the CUDA library, so both sides
can consume the same inputs.  The one piece of sampling here is the simulated
*draft model's* own sampler (it proposes y_i ~ q_i; the draft model is the
component before verification, "Speculative decoding: accelerate LLM generation
without changing its answers", section 2: "the draft samples a block y_1:k
sequentially from q").  It is written independently with a sort and a
cumulative sum in fp64.

Workloads (shapes and distributions as the method's benchmark configurations
describe them; "N(m, s^2)" is an i.i.d. normal per entry):

  small_fp32      B=1, k=5, V=1024, fp32 target logits N(0, 2^2), draft logits
                  = target + N(0, 0.5^2), T=1; contiguous KV, prefix 32.
  paged_bf16      B=8, k=4, V=32000, bf16, draft = target + N(0, 0.5^2),
                  T_b ~ U[0.5, 1.2], S_b ~ U[1, 2048], forced scenarios per request.
  ragged_probs    B=64, k_b ~ U{1..8}, V=128256, bf16 target N(0, 3^2), fp32
                  draft probabilities softmax(target + N(0, 1)), T=0.8, top-p 0.95.
  verify_b64_k4   B=64, k=4, V=128256, bf16 target N(0, 3^2), bf16 draft logits
                  target + N(0, 1), T=0.8, top-p 0.95 (top_p=1 variant too).
  greedy_shared   B=256, k=4, V=151936, bf16, draft = target + N(0, 1); even b
                  T=0, odd b T=1; groups of 4 share a 1024-token prefix.
  sweep           B in {1,16,64,256,1024}, k=8, V in {32000,128256,256000},
                  draft noise sigma in {0.25, 1, 4}, T=1.
"""

from __future__ import annotations

import numpy as np

WORKLOADS = ("small_fp32", "paged_bf16", "ragged_probs", "verify_b64_k4",
             "greedy_shared", "sweep")


# --------------------------------------------------------------------------- #
# helpers
# --------------------------------------------------------------------------- #
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (finite inputs, +-inf)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    finite = np.isfinite(np.asarray(x, dtype=np.float32))
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    r = np.where(finite, r, u >> np.uint64(16))
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


BF16_NEG_INF = np.uint16(0xFF80)


def _draft_values(d, draft_dtype):
    return bf16_bits_to_f32(d).astype(np.float64) if draft_dtype == "bf16" \
        else np.asarray(d, np.float64)


def draft_sample(row, kind: str, T: float, top_p: float, rng) -> int:
    """The simulated draft model's own sampler: y ~ top-p(softmax(row / T)).

    T = 0 samples uniformly among the tied maxima.  Written with a descending
    sort and a cumulative sum (independent of the verifier and the oracle).
    """
    row = np.asarray(row, np.float64)
    if T == 0.0:
        idx = np.flatnonzero(row == row.max())
        return int(idx[rng.integers(idx.size)])
    with np.errstate(divide="ignore"):
        z = (np.log(row) if kind == "probs" else row) / T
    w = np.exp(z - z.max())
    order = np.argsort(-w, kind="stable")
    ws = w[order] / w.sum()
    if top_p < 1.0:
        c = np.cumsum(ws)
        cut = int(np.searchsorted(c, top_p * c[-1]))          # first index reaching top_p
        cut = min(cut, ws.size - 1)
        # keep every token tied with the last kept value
        last = ws[cut]
        cut = int(np.searchsorted(-ws, -last, side="right")) - 1
        ws = ws[:cut + 1]
        order = order[:cut + 1]
    c = np.cumsum(ws)
    r = rng.random() * c[-1]
    j = min(int(np.searchsorted(c, r, side="right")), c.size - 1)
    return int(order[j])


def _sample_tokens(inp, rng):
    B, kmax = inp["tokens"].shape
    for b in range(B):
        for i in range(int(inp["k"][b])):
            row = _draft_values(inp["draft"][b, i], inp["draft_dtype"])
            inp["tokens"][b, i] = draft_sample(row, inp["draft_kind"],
                                               float(inp["temperature"][b]),
                                               float(inp["top_p"][b]), rng)


def _base(B, kmax, V, target_dtype, draft_dtype, draft_kind, seed):
    return dict(B=B, kmax=kmax, V=V, target_dtype=target_dtype, draft_dtype=draft_dtype,
                draft_kind=draft_kind, seed=int(seed),
                tokens=np.zeros((B, kmax), np.int32),
                k=np.full(B, kmax, np.int32),
                temperature=np.ones(B, np.float32),
                top_p=np.ones(B, np.float32),
                request_id=np.arange(B, dtype=np.uint32),
                seq_len=np.zeros(B, np.int32))


def _normal_bf16(rng, shape, sd):
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(sd))


# --------------------------------------------------------------------------- #
# workloads
# --------------------------------------------------------------------------- #
def small_fp32(B=1, k=5, V=1024, index=0):
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, k, V, "f32", "f32", "logits", 2000 + index)
    t = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(2.0)
    inp["target"] = t
    inp["draft"] = (t[:, :k] + rng.standard_normal((B, k, V), dtype=np.float32)
                    * np.float32(0.5)).astype(np.float32)
    inp["seq_len"][:] = 32
    inp["kv"] = dict(layout="contig", layers=2, heads=4, head_dim=64, dtype="f32")
    _sample_tokens(inp, np.random.default_rng(3000 + index))
    return inp


def paged_bf16(B=8, k=4, V=32000, index=1, forced=True):
    """Forced scenarios (request b): b < 4 rejects at position b; b = 4 makes the
    rejected tail start on a block's first slot; b = 5 leaves the kept prefix one
    slot into a fresh block; b = 6 accepts everything (q = p); others natural."""
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, k, V, "bf16", "bf16", "logits", 2000 + index)
    t = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(2.0)
    d = t[:, :k] + rng.standard_normal((B, k, V), dtype=np.float32) * np.float32(0.5)
    inp["target"] = to_bf16_bits(t)
    inp["draft"] = to_bf16_bits(d)
    inp["temperature"] = rng.uniform(0.5, 1.2, B).astype(np.float32)
    inp["seq_len"] = rng.integers(1, 2049, B).astype(np.int32)
    inp["kv"] = dict(layout="paged", block_size=16, layers=4, heads=8, head_dim=128,
                     dtype="bf16")
    reject_at = {}
    if forced:
        for b in range(B):
            if b < min(4, k):
                reject_at[b] = b
            elif b == 4:
                reject_at[b] = 2
                S = int(inp["seq_len"][b])
                inp["seq_len"][b] = max(13, S - (S + 1 + 2) % 16)       # S+1+2 = 0 mod 16
            elif b == 5:
                reject_at[b] = 1
                S = int(inp["seq_len"][b])
                inp["seq_len"][b] = max(15, S - (S + 1 + 1 - 1) % 16)   # S+1+1 = 1 mod 16
            elif b == 6:
                reject_at[b] = None                                     # q = p everywhere
        for b, r in reject_at.items():
            last = k if r is None else r
            inp["draft"][b, :last] = inp["target"][b, :last]
    _sample_tokens(inp, np.random.default_rng(3000 + index))
    for b, r in reject_at.items():
        if r is not None:
            inp["target"][b, r, inp["tokens"][b, r]] = BF16_NEG_INF     # p(y_r) = 0
    inp["forced_reject_at"] = reject_at
    return inp


def ragged_probs(B=64, kmax=8, V=128256, index=2, top_p=0.95):
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, kmax, V, "bf16", "f32", "probs", 2000 + index)
    t = rng.standard_normal((B, kmax + 1, V), dtype=np.float32) * np.float32(3.0)
    dl = t[:, :kmax].astype(np.float64) + rng.standard_normal((B, kmax, V))
    dl -= dl.max(axis=-1, keepdims=True)
    e = np.exp(dl)
    inp["target"] = to_bf16_bits(t)
    inp["draft"] = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    inp["k"] = rng.integers(1, kmax + 1, B).astype(np.int32)
    inp["temperature"][:] = 0.8
    inp["top_p"][:] = top_p
    inp["seq_len"] = rng.integers(128, 8193, B).astype(np.int32)
    inp["kv"] = dict(layout="paged", block_size=16, layers=32, heads=8, head_dim=128,
                     dtype="bf16")
    _sample_tokens(inp, np.random.default_rng(3000 + index))
    return inp


def verify_b64_k4(B=64, k=4, V=128256, index=5, top_p=0.95, sample_tokens=True):
    """The throughput workload: bf16 target N(0,3^2), bf16 draft logits
    target + N(0,1), T=0.8, top-p 0.95 on p and q, S_b ~ U[128, 8192]."""
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, k, V, "bf16", "bf16", "logits", 2000 + index)
    t = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(3.0)
    d = t[:, :k] + rng.standard_normal((B, k, V), dtype=np.float32)
    inp["target"] = to_bf16_bits(t)
    inp["draft"] = to_bf16_bits(d)
    inp["temperature"][:] = 0.8
    inp["top_p"][:] = top_p
    inp["seq_len"] = rng.integers(128, 8193, B).astype(np.int32)
    inp["kv"] = dict(layout="paged", block_size=16, layers=32, heads=8, head_dim=128,
                     dtype="bf16")
    if sample_tokens:
        _sample_tokens(inp, np.random.default_rng(3000 + index))
    return inp


def greedy_shared(B=256, k=4, V=151936, index=3, group=4, prefix=1024):
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, k, V, "bf16", "bf16", "logits", 2000 + index)
    t = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(3.0)
    d = t[:, :k] + rng.standard_normal((B, k, V), dtype=np.float32)
    inp["target"] = to_bf16_bits(t)
    inp["draft"] = to_bf16_bits(d)
    inp["temperature"] = np.where(np.arange(B) % 2 == 0, 0.0, 1.0).astype(np.float32)
    inp["seq_len"] = (prefix + rng.integers(0, 32, B)).astype(np.int32)
    inp["kv"] = dict(layout="paged", block_size=16, layers=28, heads=4, head_dim=128,
                     dtype="bf16", share_group=group, shared_prefix=prefix)
    _sample_tokens(inp, np.random.default_rng(3000 + index))
    return inp


def sweep(B=16, V=32000, sigma=1.0, k=8, index=4):
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, k, V, "bf16", "bf16", "logits", 2000 + index)
    t = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(3.0)
    d = t[:, :k] + rng.standard_normal((B, k, V), dtype=np.float32) * np.float32(sigma)
    inp["target"] = to_bf16_bits(t)
    inp["draft"] = to_bf16_bits(d)
    inp["seq_len"] = rng.integers(128, 8193, B).astype(np.int32)
    inp["kv"] = dict(layout="paged", block_size=16, layers=32, heads=8, head_dim=128,
                     dtype="bf16")
    _sample_tokens(inp, np.random.default_rng(3000 + index))
    return inp


def tiny(V=8, k=3, B=256, T=1.0, top_p=1.0, seed=7, index=9, noise=1.0,
         target_dtype="f32", draft_kind="logits", draft_dtype="f32"):
    """Small-vocabulary batches for distribution tests: each request is an
    independent trial over the same rows (rows repeat across requests)."""
    rng = np.random.default_rng(1000 + index)
    inp = _base(B, k, V, target_dtype, draft_dtype, draft_kind, seed)
    t1 = rng.standard_normal((1, k + 1, V), dtype=np.float32) * np.float32(1.5)
    d1 = t1[:, :k] + rng.standard_normal((1, k, V), dtype=np.float32) * np.float32(noise)
    t = np.repeat(t1, B, axis=0)
    d = np.repeat(d1, B, axis=0)
    if draft_kind == "probs":
        e = np.exp(d.astype(np.float64) - d.max(axis=-1, keepdims=True))
        d = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    inp["target"] = to_bf16_bits(t) if target_dtype == "bf16" else t
    inp["draft"] = to_bf16_bits(d) if draft_dtype == "bf16" else d.astype(np.float32)
    inp["temperature"][:] = T
    inp["top_p"][:] = top_p
    inp["request_id"] = np.arange(B, dtype=np.uint32) + np.uint32(seed * 65537 % 100003)
    inp["seq_len"] = np.full(B, 5, np.int32)
    _sample_tokens(inp, np.random.default_rng(3000 + index + seed))
    return inp


# --------------------------------------------------------------------------- #
# token trees
# --------------------------------------------------------------------------- #
def tree_shape(shape: str, rng) -> list:
    """Parents (parent[i - 1] of node i; 0 = the root) of a named tree shape:
    'chain:k', 'binary:d' (full binary tree of depth d), 'wide:w,d' (w root
    children, each the head of a chain of depth d), 'random:n' (node i hangs
    under a uniformly chosen earlier node)."""
    kind, arg = shape.split(":")
    if kind == "chain":
        return list(range(int(arg)))
    if kind == "binary":
        par, level = [], [0]
        for _ in range(int(arg)):
            nxt = []
            for p in level:
                for _ in range(2):
                    par.append(p)
                    nxt.append(len(par))
            level = nxt
        return par
    if kind == "wide":
        w, d = (int(x) for x in arg.split(","))
        par = []
        for _ in range(w):
            par.append(0)
            for _ in range(d - 1):
                par.append(len(par))
        return par
    if kind == "random":
        return [int(rng.integers(0, i)) for i in range(1, int(arg) + 1)]
    raise ValueError(shape)


def tree_batch(B=64, V=128256, shape="binary:3", index=6, T=0.8, top_p=0.95, dtype="bf16",
               draft_kind="logits", ragged=False):
    """Token-tree verification inputs: one tree per request (the same shape,
    or ragged node counts), target rows N(0, 3^2) and draft rows target +
    N(0, 1) per node, children drawn i.i.d. from the draft's own top-p
    distribution at their parent."""
    rng = np.random.default_rng(1000 + index)
    par = tree_shape(shape, rng)
    N = len(par)
    inp = dict(B=B, N=N, V=V, target_dtype=dtype, draft_dtype="f32" if draft_kind == "probs" else dtype,
               draft_kind=draft_kind, seed=2000 + index,
               parent=np.tile(np.array(par, np.int32), (B, 1)),
               tokens=np.zeros((B, N), np.int32),
               n=np.full(B, N, np.int32),
               temperature=np.full(B, T, np.float32), top_p=np.full(B, top_p, np.float32),
               request_id=np.arange(B, dtype=np.uint32),
               seq_len=rng.integers(128, 8193, B).astype(np.int32))
    if ragged:
        inp["n"] = rng.integers(0, N + 1, B).astype(np.int32)
    t = rng.standard_normal((B, N + 1, V), dtype=np.float32) * np.float32(3.0)
    d = t + rng.standard_normal((B, N + 1, V), dtype=np.float32)
    if draft_kind == "probs":
        e = np.exp(d.astype(np.float64) - d.max(axis=-1, keepdims=True))
        inp["draft"] = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    else:
        inp["draft"] = to_bf16_bits(d) if dtype == "bf16" else d
    inp["target"] = to_bf16_bits(t) if dtype == "bf16" else t
    srng = np.random.default_rng(3000 + index)
    for b in range(B):
        for i in range(1, N + 1):
            row = _draft_values(inp["draft"][b, par[i - 1]], inp["draft_dtype"])
            inp["tokens"][b, i - 1] = draft_sample(row, draft_kind, T, top_p, srng)
    return inp


def build(name: str, **kw):
    return {"small_fp32": small_fp32, "paged_bf16": paged_bf16,
            "ragged_probs": ragged_probs, "verify_b64_k4": verify_b64_k4,
            "greedy_shared": greedy_shared, "sweep": sweep, "tiny": tiny}[name](**kw)


def padded_ld(V: int, elem_bytes: int) -> int:
    """Row stride (elements) whose byte size is a multiple of 16."""
    per = 16 // elem_bytes
    return -(-V // per) * per
