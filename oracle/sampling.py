"""Verification step of speculative decoding, written out plainly in fp64 (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources (page titles; sections as printed on the pages):
  [SD]  "Speculative decoding: accelerate LLM generation without changing its
        answers" -- section 2 "Draft, verify, correct", 3 "Why this preserves
        the target distribution", 4 "Data flow and performance trade-offs",
        5 "Reproducible toy lab", 6 "Production failures, debugging, and
        security".
  [KV]  "Walk through KV-cache updates when speculative decoding rejects some
        draft tokens" (left-to-right acceptance, first rejection ends the run).

Per request b with k_b drafts the walk is ([SD] section 2):
  for i = 0 .. k_b - 1: accept draft y_i with probability min(1, p_i(y_i)/q_i(y_i));
  the first rejection stops the walk and a correction is drawn from
  normalize(max(0, p_i - q_i)); if every draft is accepted a bonus token is
  drawn from p_{k_b}.  Both draws are exponential races argmax_x w_x / E_x,
  which sample x with probability w_x / sum(w).

Readings taken where the pages leave a step open:
  * transforms ([SD] sections 3, 4, 6: acceptance uses "the exact transformed
    distributions"): z = logit / T, or ln(prob) / T for draft probabilities;
    dist = softmax(z).  T = 0 is the limit T -> 0+: uniform over the tied
    maximum set.
  * top-k (named by [SD] section 4 among the transforms, not defined): set
    based like top-p; tau_k = the top_k-th largest entry of the transformed
    distribution (repeats counted), keep every x with dist_x >= tau_k (so
    ties at tau_k are all kept), renormalise.  Applied before top-p, to p and
    q alike; top_k <= 0 or >= V means none; no effect at T = 0.
  * top-p: set-based nucleus.  tau = the largest value t with
    sum_{x: dist_x >= t} dist_x >= top_p; keep every x with dist_x >= tau (all
    ties at tau), renormalise.  Applied to p and to q alike; no effect at T = 0.
  * accept test without division: accept iff u * q(y) < p(y); equal to
    u < min(1, p/q) for q(y) > 0.  q(y) = 0 cannot happen for a proposal drawn
    from q ([SD] section 5, variation 2); it is flagged ST_Q_ZERO and the rule
    then accepts iff p(y) > 0.
  * a rejected row whose residual is numerically empty samples from p and is
    flagged ST_RESIDUAL_EMPTY.
  * invalid input (NaN, +inf, a row with no support, bad T / top_p / k / token)
    ends the request: accepted = -1, nothing emitted, ST_BAD_INPUT.
  * absolute position of the token decided by row i: pos = S_b + 1 + i, where
    S_b is the cache length before the pass and the pending token sits at S_b.
  * end of sequence and output caps ([CV] paragraph 5 lists both among the
    cases to test): an ACCEPTED draft equal to the request's EOS id ends the
    request there (it is emitted, no correction or bonus follows; ST_EOS); a
    cap of c tokens per call stops the walk once c accepted drafts are emitted
    (ST_CAPPED); a correction or bonus is emitted only while the cap allows.
    A cap below 1 is bad input.
  * repetition penalty ([SD] sections 4 and 6 name it, give no formula): the
    CTRL rule on the logits of the request's history ids plus the drafts before
    row i, in fp32, rounded back to bf16 for bf16 rows; target and draft logit
    rows alike; probability drafts are taken as given.  theta must be a finite
    number > 0 (1: no penalty), else bad input.
  * token trees ([CV] paragraphs 3 and 5 name tree verification and branch
    switches, not the law): the children of the current node are tested in
    ascending order, each against the running residual of p (a rejection
    replaces p_r by normalize(max(0, p_r - q))); the first accepted child
    becomes the current node; when all are rejected the correction comes from
    the last residual; a node without children gets the bonus.  Sibling rank r
    is the accept uniform's slot, so a chain is the linear walk exactly.
"""

from __future__ import annotations

import numpy as np

from . import philox

ST_Q_ZERO = 1
ST_BAD_INPUT = 2
ST_RESIDUAL_EMPTY = 4
ST_TIMEOUT = 8
ST_EOS = 16
ST_CAPPED = 32


# --------------------------------------------------------------------------- #
# input decoding
# --------------------------------------------------------------------------- #
def decode_bf16(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> fp64 values (bf16 is the top half of fp32)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """fp32 values -> the nearest bfloat16 (ties to even), returned as fp64.
    bfloat16 is the upper half of an fp32 word; infinities and NaN keep their
    class."""
    f = np.atleast_1d(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    r = np.where(np.isinf(f), u >> np.uint64(16), r)
    r = np.where(np.isnan(f), np.uint64(0x7FC0), r)
    return decode_bf16(r.astype(np.uint16))


def repetition_penalty(row: np.ndarray, ids, theta: float, dtype: str) -> np.ndarray:
    """Repetition penalty on the logits of the tokens in `ids` (a set; ids
    outside [0, V) are ignored).  [SD] section 4 ("When it wins") counts
    repetition penalties among the transforms that p and q are taken after,
    and section 6 requires draft and target to apply the same ones; the pages
    give no formula, so this takes the usual one (Keskar et al., "CTRL",
    2019): a logit l > 0 becomes l / theta, any other l becomes l * theta.
    Readings: applied to target and draft logit rows alike, before the
    temperature, in fp32 (the rows' arithmetic), and a bf16 row keeps the
    result rounded back to bf16 (ties to even)."""
    out = np.array(row, dtype=np.float64, copy=True)
    th = np.float32(theta)
    V = out.shape[-1]
    for t in sorted({int(i) for i in ids if 0 <= int(i) < V}):
        l = np.float32(out[t])
        v = np.float32(l / th) if l > 0 else np.float32(l * th)
        out[t] = float(round_bf16(v)[0]) if dtype == "bf16" else float(v)
    return out


def decode(values, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return decode_bf16(values)
    if dtype == "f32":
        return np.asarray(values, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def row_is_valid(row: np.ndarray, kind: str) -> bool:
    """A row the walk can read: no NaN, no +inf, some support ([SD] section 6,
    "numerical edge cases"; reading: such rows are reported, never sampled)."""
    if np.isnan(row).any() or np.isposinf(row).any():
        return False
    if kind == "probs":
        return bool((row >= 0).all() and (row > 0).any())
    return bool(np.isfinite(row).any())


# --------------------------------------------------------------------------- #
# transforms  ([SD] sections 3, 4, 6)
# --------------------------------------------------------------------------- #
def greedy_limit(row: np.ndarray) -> np.ndarray:
    """softmax(row / T) as T -> 0+: uniform over {x : row_x = max row}."""
    support = row == row.max()
    return support / support.sum()


def softmax_T(row: np.ndarray, kind: str, T: float) -> np.ndarray:
    """Temperature transform followed by a max-shifted softmax ([SD] section 6:
    "use stable softmax/log-probability calculations")."""
    with np.errstate(divide="ignore"):
        z = (np.log(row) if kind == "probs" else row) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def nucleus(dist: np.ndarray, top_p: float):
    """Set-based top-p (reading; the pages name top-p without defining it).

    Returns (filtered distribution, kept mask, tau, margin).  tau is the
    largest distinct value t of dist with mass{dist >= t} >= top_p; kept =
    dist >= tau.  margin = distance of top_p to the nearer edge of the step
    of the cumulative mass at tau (how close the boundary decision was).
    """
    if top_p >= 1.0:
        return dist, dist > 0, float(dist[dist > 0].min()), np.inf
    vals, counts = np.unique(dist, return_counts=True)        # ascending
    vals, counts = vals[::-1], counts[::-1]                    # descending
    cum = np.cumsum(vals * counts)                             # mass of {dist >= vals[j]}
    hit = np.nonzero(cum >= top_p)[0]
    tau = float(vals[hit[0]]) if hit.size else float(vals[vals > 0].min())
    j = int(hit[0]) if hit.size else len(vals) - 1
    margin = min(cum[j] - top_p, top_p - (cum[j - 1] if j else 0.0))
    kept = dist >= tau
    out = np.where(kept, dist, 0.0)
    return out / out.sum(), kept, tau, float(abs(margin))


def top_k_set(dist: np.ndarray, top_k: int) -> np.ndarray:
    """Set-based top-k (reading; the pages name top-k without defining it):
    tau_k = the top_k-th largest entry of dist, repeats counted; keep every x
    with dist_x >= tau_k (all ties at tau_k) and dist_x > 0."""
    tau = np.sort(dist)[::-1][top_k - 1]
    return (dist >= tau) & (dist > 0)


def transform(row: np.ndarray, kind: str, T: float, top_p: float, top_k: int = 0):
    """The decoding transform applied identically to target and draft rows:
    temperature and softmax, then top-k (0 < top_k < V), then top-p on the
    renormalised top-k distribution.

    Returns (dist, info) where info holds the kept mask and the kept fraction of
    the pre-filter mass (1 when nothing is filtered).
    """
    if T == 0.0:
        dist = greedy_limit(row)
        return dist, {"kept": dist > 0, "kept_mass": 1.0, "margin": np.inf}
    dist = softmax_T(row, kind, T)
    base, kept = dist, dist > 0
    if 0 < top_k < dist.size:
        kept = top_k_set(dist, top_k)
        base = np.where(kept, dist, 0.0)
        base = base / base.sum()
    if top_p < 1.0:
        filt, kept, _, margin = nucleus(base, top_p)
        return filt, {"kept": kept, "kept_mass": float(dist[kept].sum()), "margin": margin}
    if base is not dist:
        return base, {"kept": kept, "kept_mass": float(dist[kept].sum()), "margin": np.inf}
    return dist, {"kept": kept, "kept_mass": 1.0, "margin": np.inf}


# --------------------------------------------------------------------------- #
# the acceptance law  ([SD] sections 2, 3, 5)
# --------------------------------------------------------------------------- #
def accept_probability(p_y: float, q_y: float) -> float:
    """min(1, p(y)/q(y)) ([SD] section 2)."""
    return 1.0 if q_y <= p_y else p_y / q_y


def accepted_mass(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """q(x) a(x) = min(q(x), p(x)) ([SD] section 3)."""
    return np.minimum(p, q)


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Unfilled target mass max(0, p - q) ([SD] section 3)."""
    return np.maximum(0.0, p - q)


def accepts(u: float, p_y: float, q_y: float) -> bool:
    """Accept iff u * q(y) < p(y) -- u < min(1, p/q) without a division."""
    return u * q_y < p_y


def exponential_race(w: np.ndarray, E: np.ndarray) -> int:
    """argmax_x w_x / E_x with E_x ~ Exp(1) i.i.d.: a draw from w / sum(w).

    Ties go to the lowest index (np.argmax returns the first maximum).
    """
    with np.errstate(divide="ignore", invalid="ignore"):
        keys = np.where(w > 0, w / E, 0.0)
    return int(np.argmax(keys))


# --------------------------------------------------------------------------- #
# one request, left to right  ([SD] section 2, [KV])
# --------------------------------------------------------------------------- #
def verify_request(target_rows, draft_rows, tokens, k, T, top_p, draft_kind,
                   seed, request_id, seq_len, force=None, keep_rows=False, eos=-1, cap=None,
                   rep=None, top_k=0):
    """Run the walk for one request on decoded fp64 rows.

    target_rows [>= k+1][V], draft_rows [>= k][V], tokens [>= k] (ints).
    force: optional {row: bool} that overrides the accept decision of a row
    (the parity harness uses it to follow a counted near-tie flip).
    eos: end-of-sequence token id (< 0: none); cap: most tokens to emit (None:
    no cap).  rep: optional (theta, history ids, target dtype, draft dtype):
    row i's logits get the repetition penalty for history + tokens[:i]
    (probability drafts are taken as given).  top_k: keep the top_k largest
    entries of p and of q before top-p (<= 0 or >= V: no top-k).
    Returns a dict: accepted (-1 on bad input), tokens (emitted list), status,
    rows (per-row record: p_y, q_y, u, accept, kept masses, and p/q if keep_rows).
    """
    force = force or {}
    V = target_rows.shape[-1]
    status = 0
    rows = []
    T = float(np.float32(T))
    top_p = float(np.float32(top_p))
    bad = dict(accepted=-1, tokens=[], status=ST_BAD_INPUT, rows=rows)
    if k < 0 or k > len(tokens):
        return bad
    if not (T >= 0.0) or not (0.0 < top_p <= 1.0):
        return bad
    if cap is not None and cap < 1:
        return bad
    if rep is not None and not (0.0 < float(np.float32(rep[0])) < np.inf):
        return bad
    for i in range(k + 1):
        if cap is not None and i == cap:           # c accepted drafts emitted: stop
            return dict(accepted=i, tokens=[int(t) for t in tokens[:i]],
                        status=status | ST_CAPPED, rows=rows)
        pos = int(seq_len) + 1 + i
        trow = target_rows[i]
        if rep is not None:
            trow = repetition_penalty(trow, list(rep[1]) + [int(t) for t in tokens[:i]], rep[0], rep[2])
        if not row_is_valid(trow, "logits"):
            return bad
        p, pinfo = transform(trow, "logits", T, top_p, top_k)
        rec = {"pos": pos, "p_kept_mass": pinfo["kept_mass"], "p_margin": pinfo["margin"]}
        if keep_rows:
            rec["p"] = p
        rows.append(rec)
        if i == k:                                   # bonus row ([SD] section 2)
            E = philox.race_exponentials(seed, request_id, pos, V)
            tok = exponential_race(p, E)
            rec["race"] = {"w": p, "E": E, "token": tok}
            return dict(accepted=k, tokens=[int(t) for t in tokens[:k]] + [tok],
                        status=status, rows=rows)
        drow = draft_rows[i]
        if rep is not None and draft_kind == "logits":
            drow = repetition_penalty(drow, list(rep[1]) + [int(t) for t in tokens[:i]], rep[0], rep[3])
        y = int(tokens[i])
        if not row_is_valid(drow, draft_kind) or not (0 <= y < V):
            return bad
        q, qinfo = transform(drow, draft_kind, T, top_p, top_k)
        u = philox.accept_uniform(seed, request_id, pos)
        rec.update(q_kept_mass=qinfo["kept_mass"], q_margin=qinfo["margin"],
                   p_y=float(p[y]), q_y=float(q[y]), u=u)
        if keep_rows:
            rec["q"] = q
        if q[y] == 0.0:
            status |= ST_Q_ZERO
        ok = accepts(u, p[y], q[y])
        if i in force:
            rec["forced_from"] = ok
            ok = bool(force[i])
        rec["accept"] = ok
        if ok:
            if eos >= 0 and y == eos:                 # an accepted end of sequence
                return dict(accepted=i + 1, tokens=[int(t) for t in tokens[:i + 1]],
                            status=status | ST_EOS, rows=rows)
            continue
        # first rejection: correction from normalize(max(0, p - q))
        w = residual(p, q)
        if not (w > 0).any():
            status |= ST_RESIDUAL_EMPTY
            w = p
        E = philox.race_exponentials(seed, request_id, pos, V)
        tok = exponential_race(w, E)
        rec["race"] = {"w": w, "E": E, "token": tok}
        return dict(accepted=i, tokens=[int(t) for t in tokens[:i]] + [tok],
                    status=status, rows=rows)
    raise AssertionError("unreachable")


# --------------------------------------------------------------------------- #
# a token tree  ([CV] paragraphs 3 and 5; the per-step law of [SD] sections 2-3)
# --------------------------------------------------------------------------- #
def tree_children(parent, n):
    """children[j] = the nodes whose parent is j, in ascending node order.
    Nodes are 1..n (node 0 is the root: the pending token); parent[i - 1] is
    the parent of node i."""
    ch = {j: [] for j in range(n + 1)}
    for i in range(1, n + 1):
        ch[int(parent[i - 1])].append(i)
    return ch


def verify_tree(target_rows, draft_rows, parent, tokens, n, T, top_p, draft_kind, seed,
                request_id, seq_len, top_k=0, force=None, eos=-1, cap=None, rep=None):
    """Verify one request's token tree ([CV] paragraph 3: a tree implementation
    keeps the accepted path; paragraph 5: test tree branch switches).

    Node i (1..n) proposes tokens[i - 1] as the child of parent[i - 1] (a node
    with a lower index; 0 is the root).  target_rows[j] is the target's
    distribution of the token after node j; draft_rows[j] the draft's, from
    which j's children were drawn (independently, with repeats allowed).

    Reading (the pages name tree verification without giving its law): start
    at the root; at node j with children c_1 .. c_m (ascending) and residual
    p_1 = p_j, test c_r as in the linear walk with target p_r: accept iff
    u_r * q_j(y) < p_r(y); on rejection p_{r+1} = normalize(max(0, p_r - q_j)).
    An accepted child becomes the current node.  If every child is rejected
    the correction is drawn from p_{m+1}; at a node without children the bonus
    is drawn from p_j.  Each test is one step of the linear law with target p_r,
    so the emitted token is distributed as p_j whatever the branching.  A
    residual that becomes numerically empty stops the tests and draws from p_j
    (ST_RESIDUAL_EMPTY).  Positions: node depth d puts its token at S + d; the
    tests among j's children use pos = S + d_j + 1 and sibling rank r - 1 as
    the uniform's slot; the correction or bonus after node j uses pos = S +
    d_j + 1.  A chain-shaped tree is the linear walk exactly.
    End of sequence and output caps as in the linear walk ([CV] paragraph 5):
    an accepted child whose token is the EOS id ends the request (ST_EOS); once
    cap children are accepted the walk stops (ST_CAPPED); either way no
    correction or bonus follows.  A cap below 1 is bad input.
    rep: optional (theta, history ids, target dtype, draft dtype): the rows of
    node j get the repetition penalty for the history plus the tokens of the
    accepted path up to and including j (as row i of the linear walk does for
    y_0 .. y_{i-1}).
    force: optional {(node, rank): bool} overriding an accept decision.
    Returns accepted (path length, -1 on bad input), path (node ids), tokens
    (path tokens then the correction or bonus), status, and per-test records.
    """
    force = force or {}
    V = target_rows.shape[-1]
    T = float(np.float32(T))
    top_p = float(np.float32(top_p))
    recs = []
    bad = dict(accepted=-1, path=[], tokens=[], status=ST_BAD_INPUT, tests=recs)
    if not (T >= 0.0) or not (0.0 < top_p <= 1.0) or n < 0:
        return bad
    if cap is not None and cap < 1:
        return bad
    if rep is not None and not (0.0 < float(np.float32(rep[0])) < np.inf):
        return bad
    for i in range(1, n + 1):
        if not (0 <= int(parent[i - 1]) < i) or not (0 <= int(tokens[i - 1]) < V):
            return bad
    ch = tree_children(parent, n)
    status = 0
    cur, depth, path = 0, 0, []
    while True:
        pos = int(seq_len) + depth + 1
        trow = target_rows[cur]
        ids = None
        if rep is not None:
            ids = list(rep[1]) + [int(tokens[j - 1]) for j in path]
            trow = repetition_penalty(trow, ids, rep[0], rep[2])
        if not row_is_valid(trow, "logits"):
            return bad
        p, pinfo = transform(trow, "logits", T, top_p, top_k)
        kids = ch[cur]
        if not kids:                                   # bonus after a leaf
            E = philox.race_exponentials(seed, request_id, pos, V)
            tok = exponential_race(p, E)
            recs.append({"node": cur, "race": {"w": p, "E": E, "token": tok},
                         "p_margin": pinfo["margin"]})
            return dict(accepted=len(path), path=path,
                        tokens=[int(tokens[j - 1]) for j in path] + [tok], status=status,
                        tests=recs)
        drow = draft_rows[cur]
        if rep is not None and draft_kind == "logits":
            drow = repetition_penalty(drow, ids, rep[0], rep[3])
        if not row_is_valid(drow, draft_kind):
            return bad
        q, qinfo = transform(drow, draft_kind, T, top_p, top_k)
        pr = p
        nxt = None
        for r, j in enumerate(kids):
            y = int(tokens[j - 1])
            u = philox.accept_uniform(seed, request_id, pos, r)
            if q[y] == 0.0:
                status |= ST_Q_ZERO
            ok = bool(accepts(u, pr[y], q[y]))
            rec = {"node": j, "parent": cur, "rank": r, "p_y": float(pr[y]), "q_y": float(q[y]), "u": u,
                   "p_margin": pinfo["margin"], "q_margin": qinfo["margin"]}
            if (j, r) in force:
                rec["forced_from"] = ok
                ok = bool(force[(j, r)])
            rec["accept"] = ok
            recs.append(rec)
            if ok:
                nxt = j
                break
            w = residual(pr, q)
            if not (w > 0).any():
                status |= ST_RESIDUAL_EMPTY
                pr = None
                break
            pr = w / w.sum()
        if nxt is not None:
            path.append(nxt)
            cur, depth = nxt, depth + 1
            stop = ST_EOS if (eos >= 0 and int(tokens[nxt - 1]) == eos) else \
                ST_CAPPED if (cap is not None and depth == cap) else 0
            if stop:
                return dict(accepted=depth, path=path, tokens=[int(tokens[j - 1]) for j in path],
                            status=status | stop, tests=recs)
            continue
        wr = p if pr is None else pr                  # correction
        E = philox.race_exponentials(seed, request_id, pos, V)
        tok = exponential_race(wr, E)
        recs.append({"node": cur, "race": {"w": wr, "E": E, "token": tok},
                     "p_margin": pinfo["margin"], "q_margin": qinfo["margin"]})
        return dict(accepted=len(path), path=path,
                    tokens=[int(tokens[j - 1]) for j in path] + [tok], status=status, tests=recs)


def tree_rep(inp: dict, b: int):
    """The repetition-penalty option of tree request b (None without one)."""
    if inp.get("rep_penalty") is None:
        return None
    return (float(inp["rep_penalty"][b]), [int(t) for t in inp["rep_tokens"][b]],
            inp["target_dtype"], inp["draft_dtype"])


def verify_tree_batch(inp: dict, force=None):
    """verify_tree over every request of a tree workload dict: target
    [B][N+1][V], draft [B][N+1][V], parent [B][N], tokens [B][N], n [B],
    temperature, top_p, optional top_k, eos, max_new, rep_penalty with
    rep_tokens, seed, request_id, seq_len.  Returns
    accepted [B], path [B][N] and out_tokens [B][N+1] (-1 padded), num_emitted,
    status and the per-request records."""
    B, N = inp["parent"].shape
    acc = np.zeros(B, np.int32)
    path = np.full((B, N), -1, np.int32)
    out = np.full((B, N + 1), -1, np.int32)
    nem = np.zeros(B, np.int32)
    st = np.zeros(B, np.uint32)
    recs = []
    for b in range(B):
        nb = int(inp["n"][b])
        if not (0 <= nb <= N):
            r = dict(accepted=-1, path=[], tokens=[], status=ST_BAD_INPUT, tests=[])
        else:
            tr = decode(inp["target"][b, :nb + 1], inp["target_dtype"])
            dr = decode(inp["draft"][b, :nb + 1], inp["draft_dtype"])
            r = verify_tree(tr, dr, inp["parent"][b], inp["tokens"][b], nb,
                            inp["temperature"][b], inp["top_p"][b], inp["draft_kind"],
                            inp["seed"], int(inp["request_id"][b]), int(inp["seq_len"][b]),
                            top_k=int(inp["top_k"][b]) if inp.get("top_k") is not None else 0,
                            force=(force or {}).get(b),
                            eos=int(inp["eos"][b]) if inp.get("eos") is not None else -1,
                            cap=int(inp["max_new"][b]) if inp.get("max_new") is not None else None,
                            rep=tree_rep(inp, b))
        acc[b] = r["accepted"]
        st[b] = r["status"]
        path[b, :len(r["path"])] = r["path"]
        out[b, :len(r["tokens"])] = r["tokens"]
        nem[b] = len(r["tokens"])
        recs.append(r)
    return dict(accepted=acc, path=path, out_tokens=out, num_emitted=nem, status=st,
                records=recs)


def request_options(inp: dict, b: int) -> dict:
    """The optional per-request inputs of request b (top-k, EOS id, output
    cap, repetition penalty) as verify_request keywords."""
    return dict(
        top_k=int(inp["top_k"][b]) if inp.get("top_k") is not None else 0,
        eos=int(inp["eos"][b]) if inp.get("eos") is not None else -1,
        cap=int(inp["max_new"][b]) if inp.get("max_new") is not None else None,
        rep=None if inp.get("rep_penalty") is None else
        (float(inp["rep_penalty"][b]), [int(t) for t in inp["rep_tokens"][b]],
         inp["target_dtype"], inp["draft_dtype"]))


def verify_batch(inp: dict, force=None, keep_rows=False):
    """The batched verification step over every request of a workload dict.

    inp keys: target [B][kmax+1][V] (bf16 bits or fp32), target_dtype,
    draft [B][kmax][V], draft_dtype, draft_kind ('logits' | 'probs'),
    tokens [B][kmax], k [B], temperature [B], top_p [B], seed, request_id [B],
    seq_len [B]; optional top_k [B], eos [B], max_new [B], and rep_penalty [B] with
    rep_tokens [B][H] (-1 padded).  force: optional {b: {row: bool}}.
    Returns accepted [B], out_tokens [B][kmax+1] (-1 padded), num_emitted [B],
    status [B] and the per-request records.
    """
    B = inp["k"].shape[0]
    kmax = inp["tokens"].shape[1] if inp["tokens"].ndim == 2 else 0
    accepted = np.zeros(B, np.int32)
    out = np.full((B, kmax + 1), -1, np.int32)
    nemit = np.zeros(B, np.int32)
    status = np.zeros(B, np.uint32)
    recs = []
    for b in range(B):
        kb = int(inp["k"][b])
        if kb < 0 or kb > kmax:
            r = dict(accepted=-1, tokens=[], status=ST_BAD_INPUT, rows=[])
        else:
            trows = decode(inp["target"][b, :kb + 1], inp["target_dtype"])
            drows = decode(inp["draft"][b, :kb], inp["draft_dtype"]) if kb else \
                np.zeros((0, trows.shape[-1]))
            r = verify_request(trows, drows, inp["tokens"][b, :kb], kb,
                               inp["temperature"][b], inp["top_p"][b],
                               inp["draft_kind"], inp["seed"],
                               int(inp["request_id"][b]), int(inp["seq_len"][b]),
                               force=(force or {}).get(b), keep_rows=keep_rows,
                               **request_options(inp, b))
        accepted[b] = r["accepted"]
        status[b] = r["status"]
        nemit[b] = len(r["tokens"])
        out[b, :len(r["tokens"])] = r["tokens"]
        recs.append(r)
    return dict(accepted=accepted, out_tokens=out, num_emitted=nemit,
                status=status, records=recs)
