"""Pins of the sampling oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: values the
pages print, closed forms, textbook/library routines, brute force, or the law
of the emitted tokens.  A dropped term, a swapped p/q, a wrong index or sign in
the oracle fails at least one of them.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
from scipy import special, stats

from oracle import philox, sampling as S
from speculative_decoding_verification_07_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _toy():
    with open(os.path.join(GOLDEN, "toy_lab.json")) as f:
        return json.load(f)


# --------------------------------------------------------------------------- #
# section 5 toy lab: printed values
# --------------------------------------------------------------------------- #
def test_toy_lab_printed_values():
    g = _toy()
    p, q = np.array(g["p"]), np.array(g["q"])
    acc = S.accepted_mass(p, q)
    res = S.residual(p, q)
    np.testing.assert_allclose(acc, g["accepted_mass"], atol=1e-15)
    np.testing.assert_allclose(res, g["residual"], atol=1e-15)
    assert abs(res.sum() - g["reject_probability"]) < 1e-15
    np.testing.assert_allclose(res / res.sum(), g["correction_law"], atol=1e-15)
    np.testing.assert_allclose(acc + res, g["reconstructed"], atol=1e-15)
    # per-token acceptance probability a(x) = min(1, p/q)
    a = [S.accept_probability(pi, qi) for pi, qi in zip(p, q)]
    np.testing.assert_allclose(np.array(a) * q, acc, atol=1e-15)


def _toy_batch(n, seed):
    """n independent single-draft requests on the toy rows: target logits ln p,
    draft probabilities q, T = 1, y ~ q drawn by the simulated draft."""
    g = _toy()
    p, q = np.array(g["p"]), np.array(g["q"])
    rng = np.random.default_rng(seed)
    inp = dict(target=np.tile(np.log(p).astype(np.float32), (n, 2, 1)), target_dtype="f32",
               draft=np.tile(q.astype(np.float32), (n, 1, 1)), draft_dtype="f32",
               draft_kind="probs", tokens=rng.choice(3, size=(n, 1), p=q).astype(np.int32),
               k=np.ones(n, np.int32), temperature=np.ones(n, np.float32),
               top_p=np.ones(n, np.float32), seed=seed,
               request_id=np.arange(n, dtype=np.uint32), seq_len=np.zeros(n, np.int32))
    return inp, p, q


def test_toy_lab_sampled_walk():
    """Every rejection emits token 0 (the residual is [.3, 0, 0]); the acceptance
    rate is sum(min(p, q)) = 0.7; the first emitted token follows p."""
    n = 6000
    inp, p, q = _toy_batch(n, seed=11)
    r = S.verify_batch(inp)
    rej = r["accepted"] == 0
    assert (r["out_tokens"][rej, 0] == 0).all()
    rate = 1.0 - rej.mean()
    assert abs(rate - 0.7) < 5 * np.sqrt(0.21 / n)
    counts = np.bincount(r["out_tokens"][:, 0], minlength=3)
    assert stats.chisquare(counts, p * n).pvalue > 1e-3


# --------------------------------------------------------------------------- #
# section 3: the identity behind exactness
# --------------------------------------------------------------------------- #
def test_identity_min_plus_residual_is_p():
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = rng.integers(2, 50)
        p = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 3))
        q = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 3))
        q[rng.random(V) < 0.2] = 0
        total = S.accepted_mass(p, q) + S.residual(p, q)
        np.testing.assert_array_max_ulp(total, p, maxulp=1)
        # the rejection probability equals the residual total
        beta = sum(qi * S.accept_probability(pi, qi) for pi, qi in zip(p, q) if qi > 0)
        assert abs((1 - beta) - S.residual(p, q).sum()) < 1e-12 + abs(1 - q.sum())


# --------------------------------------------------------------------------- #
# transforms vs library routines and closed forms
# --------------------------------------------------------------------------- #
def test_softmax_T_matches_scipy():
    rng = np.random.default_rng(1)
    for T in (0.3, 0.8, 1.0, 2.5):
        l = rng.standard_normal(300) * 3
        l[5] = -np.inf
        np.testing.assert_allclose(S.softmax_T(l, "logits", T), special.softmax(l / T),
                                   rtol=1e-12, atol=1e-300)


def test_probs_transform_is_power_law():
    """softmax(ln q / T) = q^(1/T) / sum q^(1/T); zeros stay zero."""
    rng = np.random.default_rng(2)
    q = rng.dirichlet(np.ones(64))
    q[[3, 9]] = 0
    for T in (0.5, 0.8, 1.0, 1.7):
        want = np.power(q, 1.0 / T)
        np.testing.assert_allclose(S.softmax_T(q, "probs", T), want / want.sum(), rtol=1e-12)
    np.testing.assert_allclose(S.softmax_T(q, "probs", 1.0), q / q.sum(), rtol=1e-12)


def test_greedy_limit_is_small_T_limit():
    rng = np.random.default_rng(3)
    l = np.round(rng.standard_normal(40) * 2, 1)
    l[[4, 17]] = l.max() + 1.0          # a two-way tie at the maximum
    lim = S.greedy_limit(l)
    np.testing.assert_allclose(lim[[4, 17]], [0.5, 0.5])
    assert lim.sum() == 1.0 and (lim > 0).sum() == 2
    np.testing.assert_allclose(special.softmax(l / 1e-3), lim, atol=1e-12)


def _brute_force_nucleus(dist, top_p):
    """Smallest upward-closed token set with mass >= top_p, by enumerating all
    subsets (upward-closed: contains every token at least as probable as a member)."""
    V = dist.size
    best = None
    for mask in range(1, 1 << V):
        s = np.array([(mask >> i) & 1 for i in range(V)], bool)
        lo = dist[s].min()
        if not (s == (dist >= lo)).all():
            continue
        m = dist[s].sum()
        if m >= top_p - 1e-15 and (best is None or m < best[0]):
            best = (m, s)
    return best[1]


def test_top_p_against_brute_force():
    rng = np.random.default_rng(4)
    for trial in range(60):
        V = int(rng.integers(2, 10))
        dist = rng.dirichlet(np.ones(V))
        if trial % 3 == 0:                      # force ties
            dist = np.round(dist * 8) + 1
            dist = dist / dist.sum()
        top_p = float(np.float32(rng.uniform(0.05, 0.999)))
        _, kept, tau, margin = S.nucleus(dist, top_p)
        np.testing.assert_array_equal(kept, _brute_force_nucleus(dist, top_p))
        assert dist[kept].sum() >= top_p - 1e-15
    # top_p = 1 is the plain softmax
    l = rng.standard_normal(20)
    d, info = S.transform(l, "logits", 0.9, 1.0)
    np.testing.assert_allclose(d, special.softmax(l / 0.9), rtol=1e-12)
    assert info["kept"].all()


# --------------------------------------------------------------------------- #
# Philox4x32-10 against an independent library implementation
# --------------------------------------------------------------------------- #
_TRITON_SCRIPT = r"""
import os, json, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def _k(c0p, c1p, c2p, c3p, o0, o1, o2, o3, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    r0, r1, r2, r3 = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i),
                               tl.load(c2p + i), tl.load(c3p + i))
    tl.store(o0 + i, r0); tl.store(o1 + i, r1); tl.store(o2 + i, r2); tl.store(o3 + i, r3)

cfg = json.loads(sys.stdin.read())
out = []
for seed, ctr in zip(cfg["seeds"], cfg["ctrs"]):
    c = [torch.tensor(np.array(v, dtype=np.uint32).view(np.int32)) for v in ctr]
    o = [torch.zeros(len(ctr[0]), dtype=torch.int32) for _ in range(4)]
    _k[(1,)](*c, *o, seed, N=len(ctr[0]))
    out.append([(x.numpy().view(np.uint32)).tolist() for x in o])
print(json.dumps(out))
"""


def test_philox_matches_triton_interpreter():
    pytest.importorskip("triton")
    rng = np.random.default_rng(5)
    seeds = [0, 1, 0xFFFFFFFF, 0x123456789ABCDEF0, int(rng.integers(0, 2 ** 63))]
    n = 32
    ctrs = []
    for i in range(len(seeds)):
        c = rng.integers(0, 2 ** 32, size=(4, n), dtype=np.uint64)
        c[:, 0] = 0
        c[:, 1] = 0xFFFFFFFF
        ctrs.append(c.tolist())
    proc = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], capture_output=True,
                          text=True, input=json.dumps({"seeds": seeds, "ctrs": ctrs}),
                          timeout=600)
    if proc.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + proc.stderr[-300:])
    lib = json.loads(proc.stdout.strip().splitlines()[-1])
    for seed, ctr, want in zip(seeds, ctrs, lib):
        k0, k1 = philox.seed_key(seed)
        got = philox.philox4x32_10(*(np.array(v, np.uint64) for v in ctr), k0, k1)
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, np.array(w, np.uint32))


def test_uniform_and_exponential_maps():
    r = np.concatenate([np.array([0, 511, 512, 0xFFFFFE00, 0xFFFFFFFF], np.uint64),
                        np.arange(0, 2 ** 32, 2 ** 32 // 4096, dtype=np.uint64)])
    u = philox.uniform_from_bits(r)
    assert (u > 0).all() and (u < 1).all()
    assert u[0] == 2.0 ** -24 and u[4] == 1 - 2.0 ** -24
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)  # exact in fp32
    # moments of many Philox draws: U ~ U(0,1), E = -ln U ~ Exp(1)
    E = philox.race_exponentials(seed=99, request_id=3, pos=17, V=200_000)
    U = np.exp(-E)
    n = E.size
    assert abs(U.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    assert abs(E.mean() - 1.0) < 5 / np.sqrt(n)
    assert abs(E.var() - 1.0) < 5 * np.sqrt(8 / n)
    # distinct streams differ
    E2 = philox.race_exponentials(seed=99, request_id=3, pos=18, V=1000)
    E3 = philox.race_exponentials(seed=99, request_id=4, pos=17, V=1000)
    assert not np.allclose(E[:1000], E2) and not np.allclose(E[:1000], E3)


# --------------------------------------------------------------------------- #
# the exponential race samples normalize(w)
# --------------------------------------------------------------------------- #
def test_exponential_race_law():
    w = np.array([0.05, 0.0, 0.3, 0.15, 0.5, 0.0, 1e-3])
    n = 20000
    wins = np.zeros(w.size, int)
    for t in range(n):
        E = philox.race_exponentials(seed=1234, request_id=t, pos=7, V=w.size)
        wins[S.exponential_race(w, E)] += 1
    assert wins[1] == 0 and wins[5] == 0
    nz = w > 0
    assert stats.chisquare(wins[nz], w[nz] / w.sum() * n).pvalue > 1e-3


def test_race_tie_goes_to_lowest_index():
    w = np.array([0.0, 2.0, 1.0, 2.0])
    E = np.array([1.0, 1.0, 0.5, 1.0])        # keys 0, 2, 2, 2
    assert S.exponential_race(w, E) == 1


# --------------------------------------------------------------------------- #
# sections 2-3: the emitted law, acceptance counts, variations
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("V,T,top_p,kind", [(3, 1.0, 1.0, "logits"),
                                            (8, 0.7, 1.0, "probs"),
                                            (16, 1.3, 0.9, "logits")])
def test_emitted_token_law_chi_square(V, T, top_p, kind):
    """Given y_i ~ q_i, the token emitted at index i follows p_i (section 3)."""
    n = 5000
    inp = W.tiny(V=V, k=2, B=n, T=T, top_p=top_p, seed=21 + V, draft_kind=kind, noise=1.0)
    r = S.verify_batch(inp)
    for i in range(2):
        reach = r["num_emitted"] > i
        toks = r["out_tokens"][reach, i]
        p, _ = S.transform(inp["target"][0, i].astype(np.float64), "logits", T, top_p)
        counts = np.bincount(toks, minlength=V)
        sup = p > 0
        assert counts[~sup].sum() == 0
        assert stats.chisquare(counts[sup], p[sup] / p[sup].sum() * reach.sum()).pvalue > 1e-3


def test_expected_accepted_count_closed_form():
    """P(a >= j) = prod_{i<j} beta_i with beta_i = sum_x min(p_i, q_i) (section 3)."""
    n, k = 5000, 3
    inp = W.tiny(V=6, k=k, B=n, T=1.0, seed=31, noise=0.8)
    r = S.verify_batch(inp)
    beta = []
    for i in range(k):
        p, _ = S.transform(inp["target"][0, i].astype(np.float64), "logits", 1.0, 1.0)
        q, _ = S.transform(inp["draft"][0, i].astype(np.float64), "logits", 1.0, 1.0)
        beta.append(np.minimum(p, q).sum())
    want = sum(np.prod(beta[:j]) for j in range(1, k + 1))
    a = r["accepted"]
    assert abs(a.mean() - want) < 5 * a.std() / np.sqrt(n)
    for j in range(1, k + 1):
        frac = (a >= j).mean()
        pj = np.prod(beta[:j])
        assert abs(frac - pj) < 5 * np.sqrt(pj * (1 - pj) / n) + 1e-9


def test_variation1_q_equals_p_accepts_all_and_bonus_from_p():
    n, k, V = 4000, 2, 8
    inp = W.tiny(V=V, k=k, B=n, T=1.0, seed=41)
    inp["draft"] = inp["target"][:, :k].copy()
    rng = np.random.default_rng(0)
    p_rows = [S.transform(inp["target"][0, i].astype(np.float64), "logits", 1.0, 1.0)[0]
              for i in range(k + 1)]
    inp["tokens"] = np.stack([rng.choice(V, n, p=p_rows[i]) for i in range(k)], 1).astype(np.int32)
    r = S.verify_batch(inp)
    assert (r["accepted"] == k).all() and (r["status"] == 0).all()
    counts = np.bincount(r["out_tokens"][:, k], minlength=V)
    assert stats.chisquare(counts, p_rows[k] * n).pvalue > 1e-3


def test_variation2_zero_draft_mass_is_supplied_by_residual():
    """q(x0) = 0 while p(x0) > 0: x0 is never proposed, yet it is emitted at
    rate p(x0) through the residual (section 5, variation 2)."""
    n = 6000
    p = np.array([0.25, 0.35, 0.4])
    q = np.array([0.0, 0.5, 0.5])
    rng = np.random.default_rng(8)
    inp = dict(target=np.tile(np.log(p).astype(np.float32), (n, 2, 1)), target_dtype="f32",
               draft=np.tile(q.astype(np.float32), (n, 1, 1)), draft_dtype="f32",
               draft_kind="probs", tokens=rng.choice(3, size=(n, 1), p=q).astype(np.int32),
               k=np.ones(n, np.int32), temperature=np.ones(n, np.float32),
               top_p=np.ones(n, np.float32), seed=77,
               request_id=np.arange(n, dtype=np.uint32), seq_len=np.zeros(n, np.int32))
    r = S.verify_batch(inp)
    assert (r["status"] == 0).all()
    counts = np.bincount(r["out_tokens"][:, 0], minlength=3)
    assert stats.chisquare(counts, p * n).pvalue > 1e-3
    rej = r["accepted"] == 0
    assert (r["out_tokens"][rej, 0] == 0).all()     # residual is [0.25, 0, 0]


def test_greedy_limit_walk_brute_force():
    """T = 0 with unique maxima: accept iff y is the target argmax; the
    correction is the target argmax; the bonus is the last row's argmax."""
    rng = np.random.default_rng(9)
    B, k, V = 200, 3, 12
    t = np.stack([[rng.permutation(V).astype(np.float32) for _ in range(k + 1)] for _ in range(B)])
    d = t[:, :k].copy()
    flip = rng.random((B, k)) < 0.4
    for b, i in zip(*np.nonzero(flip)):
        d[b, i] = rng.permutation(V).astype(np.float32)
    inp = dict(target=t, target_dtype="f32", draft=d, draft_dtype="f32", draft_kind="logits",
               tokens=d.argmax(-1).astype(np.int32), k=np.full(B, k, np.int32),
               temperature=np.zeros(B, np.float32), top_p=np.full(B, 0.5, np.float32),
               seed=5, request_id=np.arange(B, dtype=np.uint32), seq_len=np.zeros(B, np.int32))
    r = S.verify_batch(inp)
    for b in range(B):
        a = 0
        while a < k and d[b, a].argmax() == t[b, a].argmax():
            a += 1
        assert r["accepted"][b] == a
        assert r["out_tokens"][b, a] == t[b, a].argmax()


# --------------------------------------------------------------------------- #
# invalid input and flags
# --------------------------------------------------------------------------- #
def test_bad_input_and_q_zero_flags():
    inp = W.tiny(V=8, k=2, B=6, seed=51)
    inp["target"][0, 0, 3] = np.nan
    inp["target"][1, 1, :] = -np.inf
    inp["draft"][1, 0] = inp["target"][1, 0]          # row 0 accepts, so row 1 is read
    inp["draft"][2, 0, 1] = np.inf
    inp["temperature"][3] = -1
    inp["tokens"][4, 0] = 99
    r = S.verify_batch(inp)
    for b in range(5):
        assert r["accepted"][b] == -1 and r["num_emitted"][b] == 0
        assert r["status"][b] == S.ST_BAD_INPUT
    # a bad row after the first rejection is never read
    inp = W.tiny(V=8, k=2, B=1, seed=53)
    inp["target"][0, 0, int(inp["tokens"][0, 0])] = -np.inf   # row 0 must reject
    inp["target"][0, 1, 2] = np.nan
    r = S.verify_batch(inp)
    assert r["accepted"][0] == 0 and r["status"][0] == 0
    # q(y) = 0 on a drawn proposal is flagged
    inp = W.tiny(V=8, k=1, B=1, seed=52, draft_kind="probs")
    y = int(inp["tokens"][0, 0])
    inp["draft"][0, 0, y] = 0.0
    r = S.verify_batch(inp)
    assert r["status"][0] & S.ST_Q_ZERO


def test_eos_and_output_cap():
    """End of sequence and output caps ([CV] paragraph 5 lists both as cases to
    test): q = p makes every proposal accepted, so the walk's stopping point
    is fixed by the EOS id and the cap alone."""
    rng = np.random.default_rng(40)
    V, k = 8, 4
    rows = rng.standard_normal((k + 1, V))
    y = np.array([3, 5, 2, 6])

    def run(**kw):
        return S.verify_request(rows, rows[:k], y, k, 1.0, 1.0, "logits", 9, 1, 100, **kw)

    r = run(eos=2)
    assert r["accepted"] == 3 and r["tokens"] == [3, 5, 2] and r["status"] == S.ST_EOS
    r = run(cap=2)
    assert r["accepted"] == 2 and r["tokens"] == [3, 5] and r["status"] == S.ST_CAPPED
    r = run(cap=4)                                   # the cap equals k: no bonus
    assert r["accepted"] == 4 and r["tokens"] == [3, 5, 2, 6] and r["status"] == S.ST_CAPPED
    full = run()
    r = run(cap=5)                                   # above k: the bonus fits
    assert r["accepted"] == 4 and r["tokens"] == full["tokens"] and len(r["tokens"]) == 5
    assert r["status"] == 0
    r = run(eos=5, cap=2)                            # EOS at the cap's last token
    assert r["accepted"] == 2 and r["tokens"] == [3, 5] and r["status"] == S.ST_EOS
    assert run(cap=0)["accepted"] == -1 and run(cap=0)["status"] == S.ST_BAD_INPUT
    # an EOS id that is proposed but rejected changes nothing: the correction follows
    t2 = rows.copy()
    t2[0, 3] = -np.inf                               # p(y_0) = 0: row 0 rejects
    r = S.verify_request(t2, rows[:k], y, k, 1.0, 1.0, "logits", 9, 1, 100, eos=3)
    r0 = S.verify_request(t2, rows[:k], y, k, 1.0, 1.0, "logits", 9, 1, 100)
    assert r["accepted"] == 0 and r["tokens"] == r0["tokens"] and r["status"] == 0
    # a bonus that happens to be the EOS id is emitted as usual
    r = run(eos=full["tokens"][-1])
    if full["tokens"][-1] not in y.tolist():
        assert r["tokens"] == full["tokens"] and r["status"] == 0


def test_repetition_penalty_closed_forms():
    """Repetition penalty ([SD] sections 4 and 6 name it; the rule is CTRL's):
    a positive logit is divided by theta, a negative one multiplied.  V = 2
    rows whose softmax after the penalty has a closed form: logits (ln 3, 0)
    with theta = 2 give p_0 = sqrt(3) / (1 + sqrt(3)); logits (-ln 2, 0) with
    theta = 3 give p_0 = (1/8) / (1 + 1/8) = 1/9 (the wrong sign rule gives
    2^(-1/3) / (1 + 2^(-1/3)) instead)."""
    def p_row(logits, theta, hist, i=0, dtype="f32"):
        rows = np.array([logits] * 3, dtype=np.float64)
        rows = np.asarray(np.float32(rows), np.float64)   # the rows' own fp32 values
        r = S.verify_request(rows, rows[:2], np.array([1, 1]), 2, 1.0, 1.0, "logits", 5, 0, 10,
                             keep_rows=True, rep=(theta, hist, dtype, dtype))
        return r["rows"][i]["p"], r

    p, r = p_row([np.log(3.0), 0.0], 2.0, [0])
    assert abs(p[0] - np.sqrt(3.0) / (1.0 + np.sqrt(3.0))) < 1e-6
    p, _ = p_row([-np.log(2.0), 0.0], 3.0, [0])
    assert abs(p[0] - 1.0 / 9.0) < 1e-6
    # history ids outside [0, V) and repeats change nothing; theta = 1 is no penalty
    p1, _ = p_row([np.log(3.0), 0.0], 2.0, [0, 0, 7, -3])
    assert abs(p1[0] - np.sqrt(3.0) / (1.0 + np.sqrt(3.0))) < 1e-6
    p, _ = p_row([np.log(3.0), 0.0], 1.0, [0, 1])
    assert abs(p[0] - 0.75) < 1e-6
    # the drafts before row i join the penalised set: with no history and
    # y_0 = 1, row 1 sees logit 0 of token 1 (unchanged by either rule) and
    # token 0 untouched, so p_0 = 3/4; proposing token 0 first penalises it
    rows = np.asarray(np.float32([[np.log(3.0), 0.0]] * 3), np.float64)
    r = S.verify_request(rows, rows[:2], np.array([0, 1]), 2, 1.0, 1.0, "logits", 5, 0, 10,
                         keep_rows=True, rep=(2.0, [], "f32", "f32"))
    assert abs(r["rows"][0]["p"][0] - 0.75) < 1e-6
    assert r["accepted"] == 2                       # q = p on every row
    assert abs(r["rows"][1]["p"][0] - np.sqrt(3.0) / (1.0 + np.sqrt(3.0))) < 1e-6
    # the same penalty on both sides keeps q = p: every proposal is accepted
    rng = np.random.default_rng(41)
    rows = rng.standard_normal((5, 16)) * 2
    y = np.array([3, 3, 9, 4])
    r = S.verify_request(rows, rows[:4], y, 4, 0.8, 1.0, "logits", 5, 2, 10,
                         rep=(1.7, [3, 4, 11], "f32", "f32"))
    assert r["accepted"] == 4 and r["tokens"][:4] == y.tolist()
    # bf16 rows keep the penalised value rounded to bf16 (ties to even):
    # 2 / 1.3 = 1.53846.. lies between 1.53125 and 1.5390625 (step 2^-7);
    # -2 * 1.3 = -2.6 between -2.59375 and -2.609375 (step 2^-6)
    out = S.repetition_penalty(np.array([2.0, -2.0, 0.5]), [0, 1], 1.3, "bf16")
    assert out.tolist() == [1.5390625, -2.59375, 0.5]
    # theta must be finite and > 0
    for bad in (0.0, -1.0, np.inf, np.nan):
        r = S.verify_request(rows, rows[:4], y, 4, 1.0, 1.0, "logits", 5, 2, 10,
                             rep=(bad, [], "f32", "f32"))
        assert r["accepted"] == -1 and r["status"] == S.ST_BAD_INPUT


def test_top_k_against_brute_force_and_closed_forms():
    """Top-k ([SD] section 4 names it; set-based reading): x is kept iff fewer
    than top_k entries are strictly larger than dist_x (a characterisation
    independent of the sort in the oracle), checked by brute force on small
    rows with many ties; top_k = 1 equals the greedy limit at any T > 0;
    top-k applies before top-p (a hand example where the order matters)."""
    rng = np.random.default_rng(43)
    for _ in range(300):
        V = int(rng.integers(2, 9))
        row = rng.integers(-3, 3, V).astype(np.float64)       # many ties
        tk = int(rng.integers(1, V))
        d, info = S.transform(row, "logits", 1.0, 1.0, tk)
        dist = S.softmax_T(row, "logits", 1.0)
        keep = np.array([(dist > dist[x]).sum() < tk for x in range(V)])
        assert (info["kept"] == keep).all()
        want = np.where(keep, dist, 0.0)
        np.testing.assert_allclose(d, want / want.sum(), rtol=0, atol=1e-15)
        assert abs(info["kept_mass"] - dist[keep].sum()) < 1e-15
        # top_k = 1: the tied maxima, uniformly
        d1, _ = S.transform(row, "logits", 0.7, 1.0, 1)
        np.testing.assert_allclose(d1, S.greedy_limit(row), rtol=0, atol=1e-15)
        # top_k <= 0 and top_k >= V filter nothing
        for off in (0, -1, V, V + 3):
            np.testing.assert_allclose(S.transform(row, "logits", 1.0, 1.0, off)[0], dist)
    # q = (0.4, 0.3, 0.2, 0.1), top_k = 3 then top_p = 0.75: the renormalised
    # top-3 masses 4/9, 3/9, 2/9 reach 0.75 after two entries -> (4/7, 3/7);
    # top-p first would keep three entries
    q = np.array([0.4, 0.3, 0.2, 0.1])
    d, info = S.transform(q, "probs", 1.0, 0.75, 3)
    np.testing.assert_allclose(d, [4 / 7, 3 / 7, 0.0, 0.0], rtol=0, atol=1e-15)
    assert abs(info["kept_mass"] - 0.7) < 1e-15
    d, _ = S.transform(q, "probs", 1.0, 0.75, 0)
    np.testing.assert_allclose(d, [4 / 9, 3 / 9, 2 / 9, 0.0], rtol=0, atol=1e-15)
    # at T = 0 top-k changes nothing
    row = np.array([1.0, 3.0, 3.0, 2.0])
    np.testing.assert_allclose(S.transform(row, "logits", 0.0, 1.0, 1)[0], [0, 0.5, 0.5, 0])


def test_top_k_walk_q_equals_p():
    """With q = p after the same top-k on both sides every proposal inside the
    top-k set is accepted, and a proposal outside it has q(y) = 0."""
    rng = np.random.default_rng(44)
    rows = rng.standard_normal((4, 12))
    order = np.argsort(-rows[0])
    y = np.array([order[0], order[1], order[2]])
    r = S.verify_request(rows, rows[:3], y, 3, 1.0, 1.0, "logits", 1, 0, 5, top_k=12 - 1)
    assert r["accepted"] == 3
    y_out = np.array([order[5], order[1], order[2]])               # rank 6 of row 0
    r = S.verify_request(rows, rows[:3], y_out, 3, 1.0, 1.0, "logits", 1, 0, 5, top_k=3)
    assert r["rows"][0]["q_y"] == 0.0 and r["status"] & S.ST_Q_ZERO


def test_tree_chain_is_the_linear_walk():
    """A chain-shaped token tree (node i the child of node i - 1) is the
    linear walk exactly: same accepted count, tokens and status bits."""
    rng = np.random.default_rng(45)
    for t in range(60):
        V, k = int(rng.integers(3, 12)), int(rng.integers(0, 5))
        rows = rng.standard_normal((k + 1, V)) * 2
        drows = rows + rng.standard_normal((k + 1, V))
        y = rng.integers(0, V, k)
        T, tp, tk = [(1.0, 1.0, 0), (0.7, 0.8, 0), (0.0, 1.0, 0), (1.2, 0.9, 3)][t % 4]
        lin = S.verify_request(rows, drows[:k], y, k, T, tp, "logits", 5 + t, 3, 40, top_k=tk)
        tree = S.verify_tree(rows, drows, np.arange(k), y, k, T, tp, "logits", 5 + t, 3, 40,
                             top_k=tk)
        assert tree["accepted"] == lin["accepted"] and tree["tokens"] == lin["tokens"]
        assert tree["status"] == lin["status"]
        assert tree["path"] == list(range(1, lin["accepted"] + 1))


def test_tree_root_law_chi_square():
    """Tree verification keeps the target law: m children drawn i.i.d. from q
    at the root, tested in turn against the running residual, then the
    correction; the first emitted token must follow p (chi-square), and the
    first child is accepted with probability sum_x min(p, q)."""
    rng = np.random.default_rng(46)
    V, m, n_trials = 6, 3, 6000
    p_logits = np.array([1.0, 0.2, -0.5, 0.8, -1.0, 0.0])
    q_logits = np.array([-0.3, 1.1, 0.4, 0.0, 0.6, -0.8])
    p = S.softmax_T(p_logits, "logits", 1.0)
    q = S.softmax_T(q_logits, "logits", 1.0)
    rows_t = np.stack([p_logits] + [np.zeros(V)] * m)
    rows_d = np.stack([q_logits] + [np.zeros(V)] * m)
    counts = np.zeros(V)
    first_acc = 0
    for t in range(n_trials):
        kids = rng.choice(V, m, p=q)
        r = S.verify_tree(rows_t, rows_d, np.zeros(m, np.int64), kids, m, 1.0, 1.0, "logits",
                          1000 + t, 7, 0)
        counts[r["tokens"][0]] += 1
        first_acc += r["path"][:1] == [1]
    exp = p * n_trials
    assert stats.chisquare(counts, exp).pvalue > 1e-3
    beta = np.minimum(p, q).sum()
    assert abs(first_acc / n_trials - beta) < 4 * np.sqrt(beta * (1 - beta) / n_trials)


def test_tree_branch_switch_and_repeated_siblings():
    """Branch switch worked by hand: root children y_1 (node 1) and y_2 (node
    2) with q = (1/2 at y_1, 1/2 at y_2) and p concentrated on y_2.  Node 1 has
    p(y_1) = 0 and is rejected; the residual max(0, p - q) normalised is 1 at
    y_2, so node 2 is accepted whatever u, and the walk continues below node 2
    (its child, node 3, with q = p there, is accepted too).  Then: a repeated
    sibling is never accepted after its twin was rejected."""
    V = 4
    NEG = -np.inf
    t_rows = np.array([[NEG, NEG, 0.0, NEG],        # root: p = y_2 only
                       [0.0, 0.0, 0.0, 0.0],
                       [0.0, 1.0, 2.0, 3.0],        # after node 2
                       [0.0, 0.0, 0.0, 0.0]])
    d_rows = np.array([[NEG, 0.0, 0.0, NEG],        # root: q = 1/2 on tokens 1 and 2
                       [0.0, 0.0, 0.0, 0.0],
                       [0.0, 1.0, 2.0, 3.0],        # node 2: q = p
                       [0.0, 0.0, 0.0, 0.0]])
    parent, tokens = np.array([0, 0, 2]), np.array([1, 2, 3])
    for seed in range(20):
        r = S.verify_tree(t_rows, d_rows, parent, tokens, 3, 1.0, 1.0, "logits", seed, 0, 10)
        assert r["path"] == [2, 3] and r["tokens"][:2] == [2, 3] and r["accepted"] == 2
        assert r["tests"][0]["accept"] is False and r["tests"][1]["p_y"] == 1.0
    rng = np.random.default_rng(47)
    for seed in range(200):
        tr, dr = rng.standard_normal((3, 5)), rng.standard_normal((3, 5))
        y = int(rng.integers(0, 5))
        r = S.verify_tree(tr, dr, np.array([0, 0]), np.array([y, y]), 2, 1.0, 1.0, "logits",
                          seed, 1, 0)
        assert r["path"] != [2]                      # the twin is never accepted


def test_tree_eos_and_cap():
    """EOS and output caps in a tree ([CV] paragraph 5): with q = p on every
    row, the first child of each node is accepted, so the walk follows the
    first children; an EOS id on that path or a cap ends it there, with no
    correction or bonus."""
    rng = np.random.default_rng(48)
    V = 12
    parent = np.array([0, 0, 1, 1, 3, 3, 5])           # first children: 1, 3, 5, 7
    tokens = np.array([4, 2, 7, 1, 9, 0, 6])
    rows = rng.standard_normal((8, V))

    def run(**kw):
        return S.verify_tree(rows, rows, parent, tokens, 7, 1.0, 1.0, "logits", 3, 0, 20, **kw)

    full = run()
    assert full["path"] == [1, 3, 5, 7] and full["status"] == 0 and len(full["tokens"]) == 5
    r = run(eos=9)                                      # node 5's token
    assert r["path"] == [1, 3, 5] and r["tokens"] == [4, 7, 9] and r["status"] == S.ST_EOS
    r = run(cap=2)
    assert r["path"] == [1, 3] and r["tokens"] == [4, 7] and r["status"] == S.ST_CAPPED
    r = run(cap=4)                                      # the cap equals the path: no bonus
    assert r["accepted"] == 4 and len(r["tokens"]) == 4 and r["status"] == S.ST_CAPPED
    r = run(cap=5)
    assert r["tokens"] == full["tokens"] and r["status"] == 0
    r = run(eos=7, cap=2)                               # EOS at the cap's last token
    assert r["path"] == [1, 3] and r["status"] == S.ST_EOS
    assert run(cap=0)["accepted"] == -1
    r = run(eos=2)                                      # a sibling off the path: no effect
    assert r["tokens"] == full["tokens"] and r["status"] == 0


def test_tree_repetition_penalty_is_the_linear_one_on_a_chain():
    """A chain-shaped tree with the repetition penalty gives the linear walk's
    result with the same penalty (the path tokens play the earlier drafts'
    role), on random cases with repeated proposals and history hits."""
    rng = np.random.default_rng(49)
    for t in range(40):
        V, k = int(rng.integers(4, 10)), int(rng.integers(1, 5))
        rows = rng.standard_normal((k + 1, V)) * 2
        drows = rows + rng.standard_normal((k + 1, V)) * 0.5
        y = rng.integers(0, min(V, 3), k)                  # repeats likely
        hist = list(rng.integers(-1, V + 2, 6))
        opt = (float(rng.choice([0.7, 1.3, 2.0])), hist, "f32", "f32")
        lin = S.verify_request(rows, drows[:k], y, k, 1.0, 1.0, "logits", 9 + t, 1, 30, rep=opt)
        tree = S.verify_tree(rows, drows, np.arange(k), y, k, 1.0, 1.0, "logits", 9 + t, 1, 30,
                             rep=opt)
        assert tree["tokens"] == lin["tokens"] and tree["status"] == lin["status"]
