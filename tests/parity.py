"""Compare the CUDA verification outputs with the fp64 oracle.

Bit-exact: accepted counts, emitted tokens, status bits.  Tolerated, counted
deviations (the fp32 path and the fp64 oracle may round a near-tie either way):
  * accept flip: the two disagree at row i and |u - p(y)/q(y)| < TOL there; the
    oracle is re-run following the GPU's decision and the rest must match.
  * race near-tie: the same row is sampled but the tokens differ and the
    oracle's key w/E of the GPU's token is within TOL (relative) of the winner.
  * top-p boundary: a disagreement at a row whose oracle top-p margin (distance
    of top_p to the edge of the cumulative-mass step) is below TOL.
Per-row probabilities (p(y), q(y), debug rows) must agree within 1e-6.

The tolerated cases are bounded, not only counted: a comparison fails when
they exceed one per 10^4 verified rows (at least one per call), and TALLY
sums them over the session (tests/conftest.py prints it at the end of the run).
"""

from __future__ import annotations

import numpy as np

from oracle import sampling as S

TOL = 1e-5
PROB_TOL = 1e-6

# session totals of the comparisons (printed by tests/conftest.py)
TALLY = dict(calls=0, requests=0, exact=0, accept_flips=0, race_ties=0, topp_boundary=0)


def tolerated_bound(rows):
    """Tolerated (counted) deviations allowed in one comparison of `rows`
    verified rows: one per 10^4 rows, at least one."""
    return max(1, int(rows) // 10000)


def _account(rep, rows, max_tolerated):
    n = rep["accept_flips"] + rep["race_ties"] + rep["topp_boundary"]
    bound = tolerated_bound(rows) if max_tolerated is None else max_tolerated
    TALLY["calls"] += 1
    TALLY["requests"] += rep["B"]
    for key in ("exact", "accept_flips", "race_ties", "topp_boundary"):
        TALLY[key] += rep[key]
    assert n <= bound, f"{n} tolerated deviations in {rows} rows (bound {bound}): {rep}"


def _oracle_request(inp, b, force=None, keep_rows=False):
    kb = int(inp["k"][b])
    tr = S.decode(inp["target"][b, :kb + 1], inp["target_dtype"])
    dr = S.decode(inp["draft"][b, :kb], inp["draft_dtype"]) if kb else np.zeros((0, tr.shape[-1]))
    return S.verify_request(tr, dr, inp["tokens"][b, :kb], kb, inp["temperature"][b],
                            inp["top_p"][b], inp["draft_kind"], inp["seed"],
                            int(inp["request_id"][b]), int(inp["seq_len"][b]),
                            force=force, keep_rows=keep_rows, **S.request_options(inp, b))


def _tokens(r, kmax):
    t = np.full(kmax + 1, -1, np.int64)
    t[:len(r["tokens"])] = r["tokens"]
    return t


def compare(inp, out, ref=None, max_tolerated=None):
    """Returns a report dict; raises AssertionError on an untolerated mismatch
    or on more tolerated deviations than tolerated_bound() allows."""
    acc = out["accepted"].cpu().numpy()
    tok = out["out_tokens"].cpu().numpy()
    nem = out["num_emitted"].cpu().numpy()
    st = out["status"].cpu().numpy().astype(np.uint32)
    ref = ref or S.verify_batch(inp)
    B = acc.shape[0]
    kmax = tok.shape[1] - 1
    rep = dict(B=B, exact=0, accept_flips=0, race_ties=0, topp_boundary=0, mismatches=[])
    for b in range(B):
        same = (acc[b] == ref["accepted"][b] and (tok[b] == ref["out_tokens"][b]).all()
                and nem[b] == ref["num_emitted"][b] and st[b] == ref["status"][b])
        if same:
            rep["exact"] += 1
            continue
        force = {}
        ok = False
        for _ in range(kmax + 2):
            r = _oracle_request(inp, b, force=force, keep_rows=True)
            if acc[b] == r["accepted"] and (tok[b] == _tokens(r, kmax)).all():
                ok = True
                break
            rows = r["rows"]
            if acc[b] != r["accepted"] and r["accepted"] >= 0 and acc[b] >= 0:
                i = min(acc[b], r["accepted"])
                rec = rows[i]
                if rec.get("p_margin", np.inf) < TOL or rec.get("q_margin", np.inf) < TOL:
                    rep["topp_boundary"] += 1
                    ok = True
                    break
                if "u" in rec and rec["q_y"] > 0 and abs(rec["u"] - rec["p_y"] / rec["q_y"]) < TOL:
                    rep["accept_flips"] += 1
                    force[i] = bool(acc[b] > i)
                    continue
                break
            if acc[b] == r["accepted"] and acc[b] >= 0:
                a = int(acc[b])
                rec = rows[a]
                if rec.get("p_margin", np.inf) < TOL or rec.get("q_margin", np.inf) < TOL:
                    rep["topp_boundary"] += 1
                    ok = True
                    break
                race = rec.get("race")
                g = int(tok[b, a])
                if race is not None and 0 <= g < race["w"].size:
                    keys = np.where(race["w"] > 0, race["w"] / race["E"], 0.0)
                    if keys[g] >= keys[race["token"]] * (1 - TOL) and \
                            (tok[b, :a] == _tokens(r, kmax)[:a]).all():
                        rep["race_ties"] += 1
                        ok = True
                        break
            break
        if not ok:
            rep["mismatches"].append(dict(b=b, gpu=(int(acc[b]), tok[b].tolist(), int(st[b])),
                                          oracle=(int(ref["accepted"][b]),
                                                  ref["out_tokens"][b].tolist(),
                                                  int(ref["status"][b]))))
    assert not rep["mismatches"], f"untolerated mismatches: {rep['mismatches'][:4]}"
    _account(rep, int((np.asarray(inp["k"]).astype(np.int64) + 1).sum()), max_tolerated)
    return rep


def compare_debug(inp, dbg, ref_rows=None):
    """Per-row accept operands: p(y), q(y) within PROB_TOL, u exact (fp32 grid)."""
    d = dbg.cpu().numpy()
    f = d.view(np.float32)
    i = d.view(np.int32)
    B = d.shape[0]
    checked = 0
    for b in range(B):
        r = _oracle_request(inp, b)
        for j, rec in enumerate(r["rows"]):
            if "u" not in rec or i[b, j, 5] not in (1, 2):
                continue
            if rec.get("p_margin", np.inf) < TOL or rec.get("q_margin", np.inf) < TOL:
                continue
            assert abs(f[b, j, 0] - rec["p_y"]) <= PROB_TOL, (b, j, f[b, j, 0], rec["p_y"])
            assert abs(f[b, j, 1] - rec["q_y"]) <= PROB_TOL, (b, j, f[b, j, 1], rec["q_y"])
            assert f[b, j, 2] == np.float32(rec["u"]), (b, j)
            assert abs(f[b, j, 3] - rec["p_kept_mass"]) <= 1e-5
            checked += 1
    return checked


# --------------------------------------------------------------------------- #
# token trees
# --------------------------------------------------------------------------- #
def _oracle_tree(inp, b, force=None):
    nb = int(inp["n"][b])
    tr = S.decode(inp["target"][b, :nb + 1], inp["target_dtype"])
    dr = S.decode(inp["draft"][b, :nb + 1], inp["draft_dtype"])
    return S.verify_tree(tr, dr, inp["parent"][b], inp["tokens"][b], nb, inp["temperature"][b],
                         inp["top_p"][b], inp["draft_kind"], inp["seed"],
                         int(inp["request_id"][b]), int(inp["seq_len"][b]),
                         top_k=int(inp["top_k"][b]) if inp.get("top_k") is not None else 0,
                         force=force,
                         eos=int(inp["eos"][b]) if inp.get("eos") is not None else -1,
                         cap=int(inp["max_new"][b]) if inp.get("max_new") is not None else None,
                         rep=S.tree_rep(inp, b))


def compare_tree(inp, out, ref=None, max_tolerated=None):
    """Tree outputs against the oracle: accepted length, path, tokens and
    status bit-exact, with the same counted tolerances as compare(): a test
    decided the other way where |u - p_r(y)/q(y)| < TOL (the oracle then
    follows the GPU's decision), a race near-tie, or a top-p boundary."""
    acc = out["accepted"].cpu().numpy()
    pth = out["path"].cpu().numpy()
    tok = out["out_tokens"].cpu().numpy()
    nem = out["num_emitted"].cpu().numpy()
    st = out["status"].cpu().numpy().astype(np.uint32)
    ref = ref or S.verify_tree_batch(inp)
    B, N = inp["parent"].shape
    rep = dict(B=B, exact=0, accept_flips=0, race_ties=0, topp_boundary=0, mismatches=[])
    for b in range(B):
        same = (acc[b] == ref["accepted"][b] and (pth[b, :N] == ref["path"][b]).all()
                and (tok[b] == ref["out_tokens"][b]).all() and nem[b] == ref["num_emitted"][b]
                and st[b] == ref["status"][b])
        if same:
            rep["exact"] += 1
            continue
        gp = [int(x) for x in pth[b, :max(acc[b], 0)]]
        force, ok = {}, False
        for _ in range(4 * N + 4):
            r = _oracle_tree(inp, b, force)
            rp = r["path"]
            rt = np.full(N + 1, -1, np.int64)
            rt[:len(r["tokens"])] = r["tokens"]
            if acc[b] == r["accepted"] and gp == rp and (tok[b] == rt).all():
                ok = True
                break
            if acc[b] < 0 or r["accepted"] < 0:
                break
            d = 0
            while d < min(len(gp), len(rp)) and gp[d] == rp[d]:
                d += 1
            if d < len(gp) or d < len(rp):          # a test decided differently
                parent = 0 if d == 0 else rp[d - 1]
                want = {gp[d] if d < len(gp) else None, rp[d] if d < len(rp) else None}
                tests = [t for t in r["tests"] if t.get("parent") == parent and "rank" in t]
                t = next((t for t in tests if t["node"] in want), None)
                if t is None:
                    break
                if t["q_y"] > 0 and abs(t["u"] - t["p_y"] / t["q_y"]) < TOL:
                    rep["accept_flips"] += 1
                    force[(t["node"], t["rank"])] = d < len(gp) and t["node"] == gp[d]
                    continue
                if t["p_margin"] < TOL or t["q_margin"] < TOL:
                    rep["topp_boundary"] += 1
                    ok = True
                break
            last = r["tests"][-1]                   # same path: the correction or bonus
            g = int(tok[b, len(gp)])
            if last.get("p_margin", np.inf) < TOL or last.get("q_margin", np.inf) < TOL:
                rep["topp_boundary"] += 1
                ok = True
                break
            race = last.get("race")
            if race is not None and 0 <= g < race["w"].size:
                keys = np.where(race["w"] > 0, race["w"] / race["E"], 0.0)
                if keys[g] >= keys[race["token"]] * (1 - TOL):
                    rep["race_ties"] += 1
                    ok = True
            break
        if not ok:
            rep["mismatches"].append(dict(b=b, gpu=(int(acc[b]), gp, tok[b].tolist(), int(st[b])),
                                          oracle=(int(ref["accepted"][b]),
                                                  ref["path"][b].tolist(),
                                                  ref["out_tokens"][b].tolist(),
                                                  int(ref["status"][b]))))
    assert not rep["mismatches"], f"untolerated mismatches: {rep['mismatches'][:4]}"
    _account(rep, int(np.asarray(inp["n"]).astype(np.int64).sum() + B), max_tolerated)
    return rep
