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
"""

from __future__ import annotations

import numpy as np

from oracle import philox, sampling as S

TOL = 1e-5
PROB_TOL = 1e-6


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


def compare(inp, out, ref=None):
    """Returns a report dict; raises AssertionError on an untolerated mismatch."""
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
