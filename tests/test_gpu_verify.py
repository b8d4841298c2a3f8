"""GPU parity of spec_verify against the fp64 oracle, through the C ABI.

Every configuration of the method's benchmark set is run at full size and
compared request by request (accepted counts, emitted tokens and status bits
bit-exact; near-tie flips counted under the rules in tests/parity.py), plus
edge cases, distribution tests and the normalised rows on small vocabularies.
"""

import os

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import sampling as S
from speculative_decoding_verification_07_gb300 import binding, device_io
from speculative_decoding_verification_07_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["cluster", "stream"])
def ver(request):
    """Every test runs on both kernels behind spec_verify: the cluster-resident
    one (the default) and the streaming one (SV_FLAG_STREAM_PATH; calls it
    does not serve stay on the cluster kernel)."""
    if not os.path.exists(binding.LIB_PATH):
        from speculative_decoding_verification_07_gb300 import build
        build.build()
    v = binding.Verifier(0)
    v.path_flags = binding.FLAG_STREAM_PATH if request.param == "stream" else 0
    yield v
    v.close()


def run(ver, inp, flags=0, debug=False, probs=False):
    dev = device_io.to_device(inp, "cuda:0")
    B, kmax, V = inp["tokens"].shape[0], inp["tokens"].shape[1], inp["target"].shape[-1]
    dbg = torch.zeros(B, kmax + 1, 8, dtype=torch.int32, device="cuda:0") if debug else None
    pp = torch.full((B, kmax + 1, V), -1.0, device="cuda:0") if probs else None
    pq = torch.full((B, max(kmax, 1), V), -1.0, device="cuda:0") if probs else None
    out = ver.verify(**dev, flags=flags, debug=dbg, probs_p=pp, probs_q=pq)
    torch.cuda.synchronize()
    assert ver.error() == 0
    return out, dbg, pp, pq


def report(name, rep):
    print(f"{name}: {rep['exact']}/{rep['B']} exact, accept flips {rep['accept_flips']}, "
          f"race near-ties {rep['race_ties']}, top-p boundary {rep['topp_boundary']}")


# --------------------------------------------------------------------------- #
# the benchmark configurations at full size
# --------------------------------------------------------------------------- #
def test_small_fp32_many_seeds(ver):
    total = dict(exact=0, B=0)
    for s in range(24):
        inp = W.small_fp32()
        inp["seed"] = 2000 + s
        inp["request_id"][:] = s
        out, dbg, _, _ = run(ver, inp, debug=True)
        rep = parity.compare(inp, out)
        parity.compare_debug(inp, dbg)
        total["exact"] += rep["exact"]
        total["B"] += rep["B"]
    assert total["exact"] == total["B"]


def test_paged_bf16_forced_scenarios(ver):
    inp = W.paged_bf16()
    out, dbg, _, _ = run(ver, inp, debug=True)
    report("paged_bf16", parity.compare(inp, out))
    parity.compare_debug(inp, dbg)
    acc = out["accepted"].cpu().numpy()
    for b, r in inp["forced_reject_at"].items():
        assert acc[b] == (inp["k"][b] if r is None else r), (b, acc[b], r)


def test_ragged_probs_top_p(ver):
    inp = W.ragged_probs()
    out, dbg, _, _ = run(ver, inp, debug=True)
    report("ragged_probs", parity.compare(inp, out))
    assert parity.compare_debug(inp, dbg) > 0


def test_top_p_boundary_outside_the_first_window(ver):
    """Rows whose top-p boundary sits in a plateau of up to 120000 tied logits.
    The kernel's first window assumes few elements below the boundary, so on
    these rows the boundary falls below it (or beyond the 256-key window) and
    the exact radix descent must decide it; b = 1 sits just inside the window."""
    V = 128256
    inp = W.paged_bf16(B=4, k=2, V=V, forced=False)
    rng = np.random.default_rng(77)
    # (top logit, plateau size, plateau logit) per request; T = 1, top_p = 0.95
    shapes = [(20.0, 120000, 6.0), (20.0, 100000, 8.0), (0.0, 3000, -9.0), None]
    for b, shape in enumerate(shapes):
        for arr, rows in (("target", 3), ("draft", 2)):
            for i in range(rows):
                if shape is None:
                    x = rng.standard_normal(V).astype(np.float32) * np.float32(3.0)
                else:
                    top, n, lvl = shape
                    x = np.full(V, -30.0, np.float32)
                    idx = rng.choice(V, n + 1, replace=False)
                    x[idx[:n]] = lvl + (0.5 if arr == "draft" and i == 1 else 0.0)
                    x[idx[n]] = top
                inp[arr][b, i] = W.to_bf16_bits(x)
    inp["temperature"][:] = 1.0
    inp["top_p"][:] = 0.95
    W._sample_tokens(inp, np.random.default_rng(3077))
    out, dbg, _, _ = run(ver, inp, debug=True)
    report("top-p plateau", parity.compare(inp, out))
    assert parity.compare_debug(inp, dbg) > 0
    # the plateau is inside the nucleus of the target's first row (b = 0, 1, 2)
    for b in range(3):
        p, info = S.transform(S.decode(inp["target"][b, 0], "bf16"), "logits", 1.0, 0.95)
        assert int(info["kept"].sum()) > 1000


@pytest.mark.parametrize("V", [4093, 128256])
def test_eos_and_output_caps(ver, V):
    """EOS ids drawn from the requests' own proposals and random output caps
    (some below k, some above, one invalid): outputs match the oracle's walk."""
    inp = W.verify_b64_k4(B=64, V=V)
    rng = np.random.default_rng(V)
    B, k = inp["tokens"].shape
    eos = np.full(B, -1, np.int32)
    pick = rng.random(B) < 0.6
    eos[pick] = inp["tokens"][pick, rng.integers(0, k, pick.sum())]
    cap = rng.integers(1, k + 3, B).astype(np.int32)
    cap[::5] = 1_000_000                            # effectively no cap
    cap[7] = 0                                      # invalid
    inp["eos"], inp["max_new"] = eos, cap
    out, dbg, _, _ = run(ver, inp, debug=True)
    rep = parity.compare(inp, out)
    report(f"eos/caps V={V}", rep)
    st = out["status"].cpu().numpy()
    acc = out["accepted"].cpu().numpy()
    assert acc[7] == -1 and st[7] == binding.ST_BAD_INPUT
    assert (st & binding.ST_EOS).any() and (st & binding.ST_CAPPED).any()
    nem = out["num_emitted"].cpu().numpy()
    assert (nem <= np.maximum(cap, 0)).all()
    # requests stopped by EOS or the cap emit exactly their accepted drafts
    stopped = (st & (binding.ST_EOS | binding.ST_CAPPED)) != 0
    assert (nem[stopped] == acc[stopped]).all()


def _add_repetition_penalty(inp, seed, H=300, thetas=(1.0, 1.1, 1.3, 2.0, 0.7)):
    """A generated history per request: random ids, some of the request's own
    proposals (so p(y) and q(y) move too), repeats, ids >= V and -1 padding."""
    rng = np.random.default_rng(seed)
    B, k = inp["tokens"].shape
    V = inp["target"].shape[-1]
    hist = rng.integers(0, V, (B, H)).astype(np.int32)
    for b in range(B):
        for i in range(k):
            if rng.random() < 0.5:
                hist[b, rng.integers(2, H - 8)] = inp["tokens"][b, i]
    hist[:, 1] = hist[:, 0]
    hist[::3, -6] = V + 11
    hist[:, -5:] = -1
    inp["rep_tokens"] = hist
    inp["rep_penalty"] = rng.choice(np.array(thetas, np.float32), B)


@pytest.mark.parametrize("name", ["bf16 logits V=128256", "fp32 logits V=1024",
                                  "fp32 probabilities V=128256", "greedy V=151936"])
def test_repetition_penalty(ver, name):
    """Repetition penalty on target and draft logits (CTRL's rule; draft
    probabilities untouched), with histories that hold the proposals, repeats
    and ignored ids; two requests with an invalid theta end as bad input."""
    if name.startswith("bf16"):
        inp = W.verify_b64_k4()
    elif name.startswith("fp32 logits"):
        inp = W.small_fp32(B=48)
        inp["temperature"][:] = 0.9
        inp["top_p"][::2] = 0.9
    elif name.startswith("fp32 prob"):
        inp = W.ragged_probs(B=32)
    else:
        inp = W.greedy_shared(B=32)
    _add_repetition_penalty(inp, 77)
    inp["rep_penalty"][3] = 0.0
    inp["rep_penalty"][5] = np.nan
    out, dbg, _, _ = run(ver, inp, debug=True)
    rep = parity.compare(inp, out)
    report(f"repetition penalty, {name}", rep)
    st = out["status"].cpu().numpy()
    assert st[3] == binding.ST_BAD_INPUT and st[5] == binding.ST_BAD_INPUT
    assert parity.compare_debug(inp, dbg) > 0
    # the penalty matters: without it some request's outcome differs
    plain = dict(inp)
    plain.pop("rep_penalty"), plain.pop("rep_tokens")
    ref = S.verify_batch(plain)
    ok = np.ones(len(st), bool)
    ok[[3, 5]] = False
    assert (ref["out_tokens"][ok] != out["out_tokens"].cpu().numpy()[ok]).any()


def test_repetition_penalty_normalised_rows(ver):
    """Every row's normalised p and q after the penalty (rows after a rejection
    processed too), bf16 rows, V = 4093."""
    inp = W.verify_b64_k4(B=16, V=4093)
    _add_repetition_penalty(inp, 78, H=64, thetas=(1.5, 3.0))
    _, _, pp, pq = run(ver, inp, flags=binding.FLAG_NO_SKIP, probs=True)
    pp, pq = pp.cpu().numpy(), pq.cpu().numpy()
    checked = 0
    for b in range(inp["k"].shape[0]):
        T, tp, th = inp["temperature"][b], inp["top_p"][b], inp["rep_penalty"][b]
        for i in range(int(inp["k"][b]) + 1):
            ids = list(inp["rep_tokens"][b]) + list(inp["tokens"][b, :i])
            row = S.repetition_penalty(S.decode(inp["target"][b, i], "bf16"), ids, th, "bf16")
            p, info = S.transform(row, "logits", T, tp)
            if info["margin"] >= parity.TOL:
                np.testing.assert_allclose(pp[b, i], p, atol=parity.PROB_TOL, rtol=0)
                checked += 1
            if i < inp["k"][b]:
                row = S.repetition_penalty(S.decode(inp["draft"][b, i], "bf16"), ids, th, "bf16")
                q, info = S.transform(row, "logits", T, tp)
                if info["margin"] >= parity.TOL:
                    np.testing.assert_allclose(pq[b, i], q, atol=parity.PROB_TOL, rtol=0)
                    checked += 1
    assert checked > 60


@pytest.mark.parametrize("name", ["bf16 V=128256 top-p 0.95", "bf16 V=128256 top-p 1",
                                  "fp32 logits V=1024", "fp32 probabilities V=128256",
                                  "bf16 plateaus V=4093"])
def test_top_k(ver, name):
    """Top-k before top-p on p and q: small k (inside the 256-value window
    below the maximum), large k (past it: the radix descent), k = 1, and values
    that mean no top-k (0, -1, V, > V)."""
    rng = np.random.default_rng(len(name))
    if name.startswith("bf16 V"):
        inp = W.verify_b64_k4(top_p=0.95 if "0.95" in name else 1.0)
    elif name.startswith("fp32 logits"):
        inp = W.small_fp32(B=48)
        inp["temperature"][:] = 0.9
        inp["top_p"][::2] = 0.9
    elif name.startswith("fp32 prob"):
        inp = W.ragged_probs(B=32)
    else:
        # integer logits: thousands of ties at every value, so the top-k
        # boundary always falls inside a tied group
        inp = W.verify_b64_k4(B=32, V=4093, top_p=0.95, sample_tokens=False)
        t = rng.integers(-4, 5, inp["target"].shape).astype(np.float32)
        inp["target"] = W.to_bf16_bits(t)
        inp["draft"] = W.to_bf16_bits(t[:, :-1] + rng.integers(-1, 2, inp["draft"].shape))
        d = W.bf16_bits_to_f32(inp["draft"])
        for b in range(d.shape[0]):                  # proposals among the draft's top values
            for i in range(d.shape[1]):
                inp["tokens"][b, i] = rng.choice(np.flatnonzero(d[b, i] >= d[b, i].max() - 1))
    B, V = inp["k"].shape[0], inp["target"].shape[-1]
    choices = np.array([1, 2, 5, 20, 50, 300, 1000, 6000, 40000, 0, -1, V, V + 7])
    inp["top_k"] = rng.choice(choices[choices < V + 8], B).astype(np.int32)
    out, dbg, _, _ = run(ver, inp, debug=True)
    rep = parity.compare(inp, out)
    report(f"top-k, {name}", rep)
    assert parity.compare_debug(inp, dbg) > 0
    plain = dict(inp)
    plain.pop("top_k")
    ref = S.verify_batch(plain)
    assert (ref["out_tokens"] != out["out_tokens"].cpu().numpy()).any()


def test_top_k_normalised_rows(ver):
    """Every row's normalised p and q after top-k and top-p (rows after a
    rejection processed too), bf16 rows, V = 4093."""
    inp = W.verify_b64_k4(B=16, V=4093)
    inp["top_k"] = np.array([1, 3, 10, 40, 100, 400, 1500, 3000] * 2, np.int32)
    inp["top_p"][8:] = 1.0
    _, _, pp, pq = run(ver, inp, flags=binding.FLAG_NO_SKIP, probs=True)
    pp, pq = pp.cpu().numpy(), pq.cpu().numpy()
    checked = 0
    for b in range(inp["k"].shape[0]):
        T, tp, kk = inp["temperature"][b], inp["top_p"][b], int(inp["top_k"][b])
        for i in range(int(inp["k"][b]) + 1):
            p, info = S.transform(S.decode(inp["target"][b, i], "bf16"), "logits", T, tp, kk)
            if info["margin"] >= parity.TOL:
                np.testing.assert_allclose(pp[b, i], p, atol=parity.PROB_TOL, rtol=0)
                checked += 1
            if i < inp["k"][b]:
                q, info = S.transform(S.decode(inp["draft"][b, i], "bf16"), "logits", T, tp, kk)
                if info["margin"] >= parity.TOL:
                    np.testing.assert_allclose(pq[b, i], q, atol=parity.PROB_TOL, rtol=0)
                    checked += 1
    assert checked > 60


@pytest.mark.parametrize("top_p", [0.95, 1.0])
def test_verify_b64_k4(ver, top_p):
    inp = W.verify_b64_k4(top_p=top_p)
    out, dbg, _, _ = run(ver, inp, debug=True)
    report(f"verify_b64_k4 top_p={top_p}", parity.compare(inp, out))
    assert parity.compare_debug(inp, dbg) > 0


@pytest.mark.parametrize("name", ["verify_b64_k4", "greedy_shared", "paged_bf16", "sweep"])
def test_streaming_and_cluster_kernels_agree(ver, name):
    """The two kernels behind spec_verify (the streaming kernel, which serves
    these calls when asked, and the cluster-resident one, the default) give the
    same outputs and the same per-row debug records."""
    inp = W.build(name) if name != "sweep" else W.sweep(B=64, V=128256, sigma=1.0)
    a, da, _, _ = run(ver, inp, flags=binding.FLAG_STREAM_PATH, debug=True)
    b, db, _, _ = run(ver, inp, flags=binding.FLAG_CLUSTER_PATH, debug=True)
    for key in ("accepted", "out_tokens", "num_emitted", "status"):
        assert torch.equal(a[key], b[key]), key
    report(f"{name} (streaming)", parity.compare(inp, a))
    sa, sb = da.cpu().numpy()[:, :, 5], db.cpu().numpy()[:, :, 5]
    both = (sa == sb) & np.isin(sa, (1, 2))
    fa, fb = da.cpu().numpy().view(np.float32), db.cpu().numpy().view(np.float32)
    assert np.abs(fa[both][:, :2] - fb[both][:, :2]).max(initial=0.0) <= 2 * parity.PROB_TOL


def test_greedy_shared(ver):
    inp = W.greedy_shared()
    out, dbg, _, _ = run(ver, inp, debug=True)
    report("greedy_shared", parity.compare(inp, out))
    assert parity.compare_debug(inp, dbg) > 0


@pytest.mark.parametrize("V,sigma", [(32000, 0.25), (32000, 4.0), (128256, 1.0), (256000, 0.25)])
def test_sweep_subset(ver, V, sigma):
    inp = W.sweep(B=16, V=V, sigma=sigma)
    out, _, _, _ = run(ver, inp)
    report(f"sweep V={V} sigma={sigma}", parity.compare(inp, out))


# --------------------------------------------------------------------------- #
# normalised rows, skipping, repeat calls
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_normalised_rows_match_oracle(ver, top_p):
    inp = W.paged_bf16(V=4093, forced=False)       # ragged tail: 4093 is not a multiple of 8
    inp["top_p"][:] = top_p
    inp["temperature"][::3] = 0.0
    _, _, pp, pq = run(ver, inp, flags=binding.FLAG_NO_SKIP, probs=True)
    pp, pq = pp.cpu().numpy(), pq.cpu().numpy()
    for b in range(inp["k"].shape[0]):
        T, tp = inp["temperature"][b], inp["top_p"][b]
        for i in range(int(inp["k"][b]) + 1):
            p, info = S.transform(S.decode(inp["target"][b, i], "bf16"), "logits", T, tp)
            if info["margin"] < parity.TOL:
                continue
            np.testing.assert_allclose(pp[b, i], p, atol=parity.PROB_TOL, rtol=0)
            if i < inp["k"][b]:
                q, info = S.transform(S.decode(inp["draft"][b, i], "bf16"), "logits", T, tp)
                if info["margin"] >= parity.TOL:
                    np.testing.assert_allclose(pq[b, i], q, atol=parity.PROB_TOL, rtol=0)


def test_skipping_does_not_change_outputs(ver):
    inp = W.verify_b64_k4(B=32, V=32000)
    a, _, _, _ = run(ver, inp)
    b, dbg, _, _ = run(ver, inp, flags=binding.FLAG_NO_SKIP, debug=True)
    for key in ("accepted", "out_tokens", "num_emitted", "status"):
        assert torch.equal(a[key], b[key])
    states = dbg.cpu().numpy()[:, :, 5]
    assert (states != binding.ROW_SKIPPED).all()


def test_repeated_calls_reuse_workspace(ver):
    inp = W.paged_bf16(V=8192, forced=False)
    first, _, _, _ = run(ver, inp)
    first = {k: v.clone() for k, v in first.items()}
    for _ in range(3):
        again, _, _, _ = run(ver, inp)
        for key in first:
            assert torch.equal(first[key], again[key])
    small = W.small_fp32()
    out, _, _, _ = run(ver, small)
    parity.compare(small, out)


def test_back_to_back_calls_without_sync(ver):
    """Calls issued back to back on one stream with no host synchronisation
    between them share the workspace safely: a call's kernel may be scheduled
    while the previous call's kernel still runs (programmatic dependent
    launch), and must still see only its own call's state."""
    a = W.verify_b64_k4(B=16, V=32000, index=11)
    b = W.verify_b64_k4(B=16, V=32000, index=12)
    da, db = device_io.to_device(a, "cuda:0"), device_io.to_device(b, "cuda:0")
    outs = [ver.verify(**(da if j % 2 == 0 else db)) for j in range(8)]
    torch.cuda.synchronize()
    assert ver.error() == 0
    report("back to back (a)", parity.compare(a, outs[0]))
    report("back to back (b)", parity.compare(b, outs[1]))
    for j in range(2, 8):
        for key in outs[j]:
            assert torch.equal(outs[j][key], outs[j % 2][key]), (j, key)


# --------------------------------------------------------------------------- #
# laws on small vocabularies
# --------------------------------------------------------------------------- #
def test_toy_lab_acceptance_rate_and_residual(ver):
    """p = [.5,.3,.2], q = [.2,.5,.3]: acceptance 0.7 and every rejection emits
    token 0 (section 5 toy lab), over 10^6 seeded trials."""
    n = 1_000_000
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.5, 0.3])
    rng = np.random.default_rng(0)
    target = torch.tensor(np.log(p), dtype=torch.float32).repeat(n, 2, 1)
    target = torch.nn.functional.pad(target, (0, 1), value=float("-inf")).cuda()
    draft = torch.nn.functional.pad(torch.tensor(q, dtype=torch.float32).repeat(n, 1, 1),
                                    (0, 1)).cuda()
    tokens = torch.tensor(rng.choice(3, size=(n, 1), p=q), dtype=torch.int32).cuda()
    out = ver.verify(target=target, draft=draft, draft_tokens=tokens, V=3,
                     temperature=torch.ones(n, device="cuda"), draft_kind="probs", seed=99,
                     request_id=torch.arange(n, dtype=torch.int32, device="cuda"))
    acc = out["accepted"].cpu().numpy()
    tok = out["out_tokens"].cpu().numpy()
    rate = acc.mean()
    assert abs(rate - 0.7) < 5 * np.sqrt(0.21 / n)
    assert (tok[acc == 0, 0] == 0).all()
    counts = np.bincount(tok[:, 0], minlength=3)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4


@pytest.mark.parametrize("V,T,top_p,kind", [(3, 1.0, 1.0, "logits"), (8, 0.7, 1.0, "probs"),
                                            (16, 1.3, 0.9, "logits")])
def test_emitted_law_chi_square(ver, V, T, top_p, kind):
    n = 200_000
    inp = W.tiny(V=V, k=2, B=n, T=T, top_p=top_p, seed=21 + V, draft_kind=kind)
    out, _, _, _ = run(ver, inp)
    tok = out["out_tokens"].cpu().numpy()
    nem = out["num_emitted"].cpu().numpy()
    for i in range(2):
        reach = nem > i
        p, _ = S.transform(inp["target"][0, i].astype(np.float64), "logits", T, top_p)
        counts = np.bincount(tok[reach, i], minlength=V)
        sup = p > 0
        assert counts[~sup].sum() == 0
        assert stats.chisquare(counts[sup], p[sup] / p[sup].sum() * reach.sum()).pvalue > 1e-4
    sub = {k: (v[:3000] if isinstance(v, np.ndarray) and v.shape[:1] == (n,) else v)
           for k, v in inp.items()}
    parity.compare(sub, {k: v[:3000] for k, v in out.items()})


# --------------------------------------------------------------------------- #
# edge cases
# --------------------------------------------------------------------------- #
def test_plain_decode_k0_and_ragged(ver):
    inp = W.ragged_probs(B=12, kmax=5, V=1000)
    inp["k"][:4] = 0
    out, _, _, _ = run(ver, inp)
    parity.compare(inp, out)
    assert (out["num_emitted"].cpu().numpy()[:4] == 1).all()


def test_greedy_ties(ver):
    inp = W.tiny(V=64, k=3, B=512, T=0.0, seed=5, target_dtype="bf16", draft_dtype="bf16")
    t = inp["target"]
    top = W.to_bf16_bits(np.float32(W.bf16_bits_to_f32(t).max() + 1.0))
    t[:, :, 7] = t[:, :, 11] = top          # tied maxima in every target row
    out, _, _, _ = run(ver, inp)
    parity.compare(inp, out)
    tok = out["out_tokens"].cpu().numpy()
    last = tok[np.arange(512), out["accepted"].cpu().numpy()]
    assert set(np.unique(last)) <= {7, 11}


def test_bad_inputs_are_flagged(ver):
    inp = W.tiny(V=40, k=2, B=8, seed=3, target_dtype="bf16", draft_dtype="bf16")
    inp["target"][0, 0, 5] = 0x7FC0                       # NaN
    inp["target"][1, 0, :] = W.BF16_NEG_INF               # no support
    inp["draft"][2, 0, 3] = 0x7F80                        # +inf
    inp["temperature"][3] = -1.0
    inp["top_p"][4] = 0.0
    inp["tokens"][5, 0] = 40                              # token id == V
    inp["k"][6] = 7                                       # k > kmax
    out, _, _, _ = run(ver, inp)
    acc = out["accepted"].cpu().numpy()
    st = out["status"].cpu().numpy()
    for b in range(7):
        assert acc[b] == -1 and st[b] == binding.ST_BAD_INPUT, b
        assert (out["out_tokens"][b] == -1).all()
    parity.compare(inp, out)


def test_q_zero_flag(ver):
    inp = W.tiny(V=16, k=1, B=4, seed=8, draft_kind="probs")
    for b in range(4):
        inp["draft"][b, 0, int(inp["tokens"][b, 0])] = 0.0
    out, _, _, _ = run(ver, inp)
    assert (out["status"].cpu().numpy() & binding.ST_Q_ZERO).all()
    parity.compare(inp, out)


def test_host_checks_launch_nothing(ver):
    inp = W.tiny(V=16, k=1, B=4, seed=8)
    dev = device_io.to_device(inp, "cuda:0")
    bad = dev["target"][:, :, 1:]                         # misaligned base pointer
    with pytest.raises(binding.SvError) as e:
        ver.verify(**{**dev, "target": bad, "V": 3})
    assert e.value.code == binding.SV_ERR_INVALID
    empty = {k: (v[:0] if isinstance(v, torch.Tensor) else v) for k, v in dev.items()}
    ver.verify(**empty)                                   # B = 0 is a no-op


def test_maximum_sizes(ver):
    """The largest k (64, every draft accepted: 65 rows per request, none
    skipped), the largest vocabulary one cluster holds (16 CTAs x 16384 =
    262144), and k = 65 refused by the host checks."""
    inp = W.sweep(B=4, V=32000, sigma=0.0, k=64)
    out, _, _, _ = run(ver, inp)
    rep = parity.compare(inp, out)
    report("k=64", rep)
    assert (out["accepted"].cpu().numpy() == 64).all()
    inp = W.sweep(B=3, V=262144, sigma=0.5, k=2)
    out, _, _, _ = run(ver, inp)
    report("V=262144", parity.compare(inp, out))
    big = W.sweep(B=1, V=64, sigma=0.5, k=65)
    dev = device_io.to_device(big, "cuda:0")
    with pytest.raises(binding.SvError) as e:
        ver.verify(**dev)
    assert e.value.code == binding.SV_ERR_INVALID


def test_bounded_wait_reports_timeout(ver):
    """Failure detection without a fault: with SV_FLAG_TEST_WITHHOLD, row 0 of
    request 0 (accepted: q = p there) never publishes its decision, so row 1
    (rejected: p(y_1) = 0) waits for it until its bound runs out.  The request
    reports SV_ST_TIMEOUT, the error word SV_ERR_TIMEOUT, every other request
    is unaffected, and the next plain call on the same handle is correct."""
    inp = W.paged_bf16()                      # request 1: q = p at row 0, rejects at row 1
    for key in ("target", "draft", "tokens"):
        inp[key][0] = inp[key][1]
    inp["temperature"][0] = inp["temperature"][1]
    ref = S.verify_batch(inp)
    assert ref["accepted"][0] == 1
    dev = device_io.to_device(inp, "cuda:0")
    out = ver.verify(**dev, flags=binding.FLAG_TEST_WITHHOLD)
    torch.cuda.synchronize()
    assert ver.error() == binding.SV_ERR_TIMEOUT
    acc = out["accepted"].cpu().numpy()
    st = out["status"].cpu().numpy()
    assert acc[0] == -1 and st[0] == binding.ST_TIMEOUT
    assert (out["out_tokens"][0] == -1).all()
    np.testing.assert_array_equal(acc[1:], ref["accepted"][1:])
    np.testing.assert_array_equal(out["out_tokens"].cpu().numpy()[1:], ref["out_tokens"][1:])
    out2 = ver.verify(**dev)
    torch.cuda.synchronize()
    assert ver.error() == 0
    np.testing.assert_array_equal(out2["accepted"].cpu().numpy(), ref["accepted"])
    np.testing.assert_array_equal(out2["out_tokens"].cpu().numpy(), ref["out_tokens"])


def _subset(inp, idx):
    """The requests idx of a workload (every per-request array sliced)."""
    out = dict(inp)
    B = inp["k"].shape[0]
    for key, v in inp.items():
        if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == B:
            out[key] = v[idx]
    out["B"] = len(idx)
    return out


@pytest.mark.parametrize("B,V,sigma", [(1024, 32000, 1.0), (256, 128256, 0.25), (64, 256000, 4.0)])
def test_sweep_full_size_sampled(ver, B, V, sigma):
    """The bandwidth sweep at full batch sizes (k = 8): the whole batch in one
    launch, 48 sampled requests compared with the oracle one by one."""
    inp = W.sweep(B=B, V=V, sigma=sigma, k=8)
    out, _, _, _ = run(ver, inp)
    idx = np.sort(np.random.default_rng(B + V).choice(B, 48, replace=False))
    sub = _subset(inp, idx)
    sub_out = {key: v[torch.as_tensor(idx, device=v.device)] for key, v in out.items()}
    report(f"sweep B={B} V={V} sigma={sigma} (48 sampled)", parity.compare(sub, sub_out))
    assert (out["accepted"].cpu().numpy() >= 0).all()


def test_all_options_together(ver):
    """Repetition penalty, top-k, top-p, EOS ids and output caps in one batch:
    the penalty comes first, then temperature, top-k and top-p; EOS and the cap
    end the walk."""
    inp = W.verify_b64_k4(B=48, V=32000)
    rng = np.random.default_rng(31)
    _add_repetition_penalty(inp, 32, H=120)
    inp["top_k"] = rng.choice(np.array([0, 3, 40, 700, 9000], np.int32), 48)
    eos = np.full(48, -1, np.int32)
    pick = rng.random(48) < 0.5
    eos[pick] = inp["tokens"][pick, rng.integers(0, 4, pick.sum())]
    inp["eos"] = eos
    inp["max_new"] = rng.integers(1, 7, 48).astype(np.int32)
    out, dbg, _, _ = run(ver, inp, debug=True)
    report("all options", parity.compare(inp, out))
    assert parity.compare_debug(inp, dbg) > 0
