"""GPU parity of spec_verify_tree and kv_commit_tree against the fp64 oracle,
through the C ABI: tree shapes (chains, full binary trees, wide roots, random
and ragged trees), dtypes and draft kinds, top-k / top-p / greedy, bad input,
a forced branch switch, the emitted law, and the accepted-path K/V gather."""

import os

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import kvcache as KC
from oracle import sampling as S
from speculative_decoding_verification_07_gb300 import binding, device_io
from speculative_decoding_verification_07_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ver():
    if not os.path.exists(binding.LIB_PATH):
        from speculative_decoding_verification_07_gb300 import build
        build.build()
    v = binding.Verifier(0)
    yield v
    v.close()


def run_tree(ver, inp):
    dev = device_io.tree_to_device(inp, "cuda:0")
    out = ver.verify_tree(**dev)
    torch.cuda.synchronize()
    assert ver.error() == 0
    return out


def report(name, rep):
    print(f"{name}: {rep['exact']}/{rep['B']} exact, accept flips {rep['accept_flips']}, "
          f"race near-ties {rep['race_ties']}, top-p boundary {rep['topp_boundary']}")


@pytest.mark.parametrize("shape,kw", [
    ("binary:3", {}),
    ("wide:4,3", {}),
    ("random:24", {"ragged": True}),
    ("binary:2", {"dtype": "f32", "V": 1024, "T": 1.0, "top_p": 1.0}),
    ("wide:3,2", {"draft_kind": "probs", "V": 32000}),
    ("random:12", {"T": 0.0, "top_p": 1.0, "V": 151936}),
    ("random:300", {"B": 8, "V": 32000}),
])
def test_tree_parity(ver, shape, kw):
    args = dict(B=48, V=128256)
    args.update(kw)
    inp = W.tree_batch(shape=shape, **args)
    out = run_tree(ver, inp)
    rep = parity.compare_tree(inp, out)
    report(f"tree {shape} {kw}", rep)
    acc = out["accepted"].cpu().numpy()
    assert (acc >= 0).all()


def test_tree_top_k(ver):
    inp = W.tree_batch(B=48, V=128256, shape="binary:3")
    rng = np.random.default_rng(5)
    inp["top_k"] = rng.choice(np.array([1, 3, 20, 300, 5000, 0]), 48).astype(np.int32)
    out = run_tree(ver, inp)
    report("tree top-k", parity.compare_tree(inp, out))


def test_chain_tree_equals_linear_kernel(ver):
    """A chain-shaped tree through spec_verify_tree gives spec_verify's outputs."""
    lin = W.verify_b64_k4(B=32)
    inp = dict(B=32, N=4, V=lin["target"].shape[-1], target_dtype="bf16", draft_dtype="bf16",
               draft_kind="logits", seed=lin["seed"],
               parent=np.tile(np.arange(4, dtype=np.int32), (32, 1)), tokens=lin["tokens"],
               n=np.full(32, 4, np.int32), temperature=lin["temperature"], top_p=lin["top_p"],
               request_id=lin["request_id"], seq_len=lin["seq_len"], target=lin["target"],
               draft=np.concatenate([lin["draft"], lin["draft"][:, :1]], axis=1))
    out_t = run_tree(ver, inp)
    dev = device_io.to_device(lin, "cuda:0")
    out_l = ver.verify(**dev)
    torch.cuda.synchronize()
    for key in ("accepted", "out_tokens", "num_emitted", "status"):
        assert torch.equal(out_t[key], out_l[key]), key


def test_tree_branch_switch_and_bad_input(ver):
    """The hand-worked branch switch (root children 1 and 2; node 1 has p = 0,
    the residual puts all mass on node 2's token, node 2's child has q = p), a
    repeated sibling, and the bad-input cases: a parent not below its node, a
    token outside [0, V), NaN on the walk, a bad temperature."""
    NEG = -np.inf
    V, B, N = 4, 8, 3
    t = np.zeros((B, N + 1, V), np.float32)
    d = np.zeros((B, N + 1, V), np.float32)
    t[:, 0] = [NEG, NEG, 0.0, NEG]
    d[:, 0] = [NEG, 0.0, 0.0, NEG]
    t[:, 2] = d[:, 2] = [0.0, 1.0, 2.0, 3.0]
    inp = dict(B=B, N=N, V=V, target_dtype="f32", draft_dtype="f32", draft_kind="logits",
               seed=3, parent=np.tile(np.array([0, 0, 2], np.int32), (B, 1)),
               tokens=np.tile(np.array([1, 2, 3], np.int32), (B, 1)), n=np.full(B, N, np.int32),
               temperature=np.ones(B, np.float32), top_p=np.ones(B, np.float32),
               request_id=np.arange(B, dtype=np.uint32), seq_len=np.full(B, 10, np.int32),
               target=t, draft=d)
    inp["parent"][4] = [0, 2, 2]          # node 2's parent is itself: bad
    inp["tokens"][5, 1] = V               # token outside [0, V): bad
    inp["target"][6, 2, 1] = np.nan       # NaN on the walk (node 2 is reached): bad
    inp["temperature"][7] = -1.0          # bad temperature
    out = run_tree(ver, inp)
    parity.compare_tree(inp, out)
    acc = out["accepted"].cpu().numpy()
    pth = out["path"].cpu().numpy()
    assert (acc[:4] == 2).all() and (pth[:4, :2] == [2, 3]).all()
    assert (acc[4:] == -1).all()
    assert (out["status"].cpu().numpy()[4:] == binding.ST_BAD_INPUT).all()


def test_tree_root_law(ver):
    """Emitted first tokens over 8192 requests sharing one root (3 children
    drawn from q) follow p (chi-square), and the first child is accepted with
    probability sum_x min(p, q)."""
    B, V, m = 8192, 6, 3
    rng = np.random.default_rng(9)
    pl = np.array([1.0, 0.2, -0.5, 0.8, -1.0, 0.0], np.float32)
    ql = np.array([-0.3, 1.1, 0.4, 0.0, 0.6, -0.8], np.float32)
    p = S.softmax_T(pl.astype(np.float64), "logits", 1.0)
    q = S.softmax_T(ql.astype(np.float64), "logits", 1.0)
    t = np.zeros((B, m + 1, V), np.float32)
    d = np.zeros((B, m + 1, V), np.float32)
    t[:, 0], d[:, 0] = pl, ql
    inp = dict(B=B, N=m, V=V, target_dtype="f32", draft_dtype="f32", draft_kind="logits",
               seed=11, parent=np.zeros((B, m), np.int32),
               tokens=rng.choice(V, (B, m), p=q).astype(np.int32), n=np.full(B, m, np.int32),
               temperature=np.ones(B, np.float32), top_p=np.ones(B, np.float32),
               request_id=np.arange(B, dtype=np.uint32), seq_len=np.zeros(B, np.int32),
               target=t, draft=d)
    out = run_tree(ver, inp)
    first = out["out_tokens"].cpu().numpy()[:, 0]
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, p * B).pvalue > 1e-3
    beta = np.minimum(p, q).sum()
    rate = (out["path"].cpu().numpy()[:, 0] == 1).mean()
    assert abs(rate - beta) < 4 * np.sqrt(beta * (1 - beta) / B)


def test_tree_commit_gathers_the_path_bit_exact(ver):
    """kv_commit_tree against the oracle's gather: the GPU's own accepted paths
    of a binary tree batch, random staged K/V, 4 layers x 8 heads x d128 bf16."""
    inp = W.tree_batch(B=16, V=4093, shape="binary:3")
    out = run_tree(ver, inp)
    acc = out["accepted"]
    B, N = inp["parent"].shape
    L, H, D, BS = 4, 8, 128, 16
    dmax = 3
    dev = ver.device
    nblk = 4 * B
    seq0 = torch.tensor(inp["seq_len"] % 1000 + 1, dtype=torch.int32, device=dev)
    max_blocks = (1000 + dmax + 2) // BS + 2
    table = torch.full((B, max_blocks), -1, dtype=torch.int32, device=dev)
    for b, s0 in enumerate(seq0.cpu().tolist()):
        table[b, s0 // BS] = 2 * b
        table[b, (s0 + dmax) // BS] = 2 * b + 1
    g = torch.Generator(device="cpu").manual_seed(4)
    stage = torch.randn(B, N + 1, L, 2, H, D, generator=g).to(torch.bfloat16).to(dev)
    kv = torch.zeros(nblk, L, 2, H, BS, D, dtype=torch.bfloat16, device=dev)
    binding.kv_commit_tree(ver.handle, acc, out["path"], seq0, table, BS, nblk, stage, kv, dmax)
    torch.cuda.synchronize()
    assert ver.error() == 0
    kv_ref = np.zeros((nblk, L, 2, H, BS, D), np.float32)
    KC.commit_copy(stage.float().cpu().numpy(), acc.cpu().numpy(), seq0.cpu().numpy(),
                   table.cpu().numpy(), kv_ref, BS, path=out["path"].cpu().numpy())
    np.testing.assert_array_equal(kv.float().cpu().numpy(), kv_ref)


def test_tree_empty_residual(ver):
    """q = p at the root and proposals outside their support: each test rejects
    (q(y) = 0, p(y) = 0) and max(0, p - q) is empty, after the last child
    (request 0, one child) or before it (request 1, two children); the
    correction then comes from p with SV_ST_RESIDUAL_EMPTY and SV_ST_Q_ZERO."""
    NEG = -np.inf
    B, V, N = 2, 4, 2
    t = np.zeros((B, N + 1, V), np.float32)
    t[:, 0] = [NEG, 0.0, 0.0, 0.0]
    inp = dict(B=B, N=N, V=V, target_dtype="f32", draft_dtype="f32", draft_kind="logits", seed=5,
               parent=np.zeros((B, N), np.int32), tokens=np.zeros((B, N), np.int32),
               n=np.array([1, 2], np.int32), temperature=np.ones(B, np.float32),
               top_p=np.ones(B, np.float32), request_id=np.arange(B, dtype=np.uint32),
               seq_len=np.full(B, 3, np.int32), target=t, draft=t.copy())
    out = run_tree(ver, inp)
    parity.compare_tree(inp, out)
    st = out["status"].cpu().numpy()
    assert (st == binding.ST_Q_ZERO | binding.ST_RESIDUAL_EMPTY).all()
    assert (out["accepted"].cpu().numpy() == 0).all()
    assert np.isin(out["out_tokens"].cpu().numpy()[:, 0], [1, 2, 3]).all()


def test_tree_repeated_calls_and_many_requests(ver):
    """The clusters take requests from a counter the handle owns, reset by the
    last cluster of each call: back-to-back calls (with a linear call between
    them) and a batch of 600 requests (many per cluster) all match the oracle."""
    a = W.tree_batch(B=600, V=1000, shape="wide:3,2", index=21)
    b = W.tree_batch(B=40, V=4093, shape="random:9", index=22, ragged=True)
    out_a = run_tree(ver, a)
    lin = W.tiny(V=64, k=3, B=16)
    ver.verify(**device_io.to_device(lin, "cuda:0"))
    out_b = run_tree(ver, b)
    out_a2 = run_tree(ver, a)
    report("600 requests", parity.compare_tree(a, out_a))
    report("after a linear call", parity.compare_tree(b, out_b))
    for key in ("accepted", "path", "out_tokens", "status"):
        assert torch.equal(out_a[key], out_a2[key]), key


def test_tree_eos_and_caps(ver):
    """EOS ids (drawn from the trees' own tokens, so some sit on accepted
    paths) and output caps from 1 to beyond the depth, one invalid cap."""
    inp = W.tree_batch(B=48, V=32000, shape="binary:3", index=23)
    rng = np.random.default_rng(24)
    B, N = inp["parent"].shape
    eos = np.full(B, -1, np.int32)
    pick = rng.random(B) < 0.7
    eos[pick] = inp["tokens"][pick, rng.integers(0, 2, pick.sum())]   # a root child's token
    inp["eos"] = eos
    inp["max_new"] = rng.integers(1, 5, B).astype(np.int32)
    inp["max_new"][::4] = 1000
    inp["max_new"][5] = 0
    out = run_tree(ver, inp)
    report("tree EOS / caps", parity.compare_tree(inp, out))
    st = out["status"].cpu().numpy()
    assert st[5] == binding.ST_BAD_INPUT
    assert (st & binding.ST_CAPPED).any() and (st & binding.ST_EOS).any()
    stopped = (st & (binding.ST_EOS | binding.ST_CAPPED)) != 0
    assert (out["num_emitted"].cpu().numpy()[stopped] == out["accepted"].cpu().numpy()[stopped]).all()


@pytest.mark.parametrize("kw", [{"V": 32000}, {"V": 4093, "dtype": "f32", "T": 1.0, "top_p": 1.0},
                                {"V": 32000, "draft_kind": "probs"}])
def test_tree_repetition_penalty(ver, kw):
    """Repetition penalty in trees: node j's rows are penalised for the history
    plus the accepted path's tokens up to j; the history holds some of the
    trees' own tokens; one request has an invalid theta."""
    inp = W.tree_batch(B=32, shape="binary:3", index=25, **kw)
    rng = np.random.default_rng(26)
    B, N = inp["parent"].shape
    hist = rng.integers(0, inp["V"], (B, 60)).astype(np.int32)
    for b in range(B):
        hist[b, :4] = inp["tokens"][b, rng.integers(0, N, 4)]
    hist[:, -3:] = -1
    inp["rep_tokens"] = hist
    inp["rep_penalty"] = rng.choice(np.array([1.0, 1.2, 2.0, 0.6], np.float32), B)
    inp["rep_penalty"][7] = np.nan
    out = run_tree(ver, inp)
    report(f"tree repetition penalty {kw}", parity.compare_tree(inp, out))
    assert out["status"].cpu().numpy()[7] == binding.ST_BAD_INPUT
    plain = dict(inp)
    plain.pop("rep_penalty"), plain.pop("rep_tokens")
    ref = S.verify_tree_batch(plain)
    ok = np.arange(B) != 7
    assert (ref["out_tokens"][ok] != out["out_tokens"].cpu().numpy()[ok]).any()
