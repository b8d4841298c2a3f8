"""GPU parity of the paged-KV kernels against the reference cache manager
(bit-exact free stack, top, refcounts, block tables, seq_lens, n_freed), and
the verify -> commit chain checked through the toy attention model."""

import os

import numpy as np
import pytest
import torch

from oracle import kvcache
from speculative_decoding_verification_07_gb300 import binding, device_io
from speculative_decoding_verification_07_gb300 import workloads as W
from tests import parity
from tests.toy_model import PagedPayload, ToyAttention

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def ver():
    if not os.path.exists(binding.LIB_PATH):
        from speculative_decoding_verification_07_gb300 import build
        build.build()
    v = binding.Verifier(0)
    yield v
    v.close()


class Pair:
    """A GPU pool and the reference pool driven with the same calls."""

    def __init__(self, ver, num_blocks, BS, B, max_blocks):
        self.ver = ver
        self.g = binding.BlockPool(ver.handle, num_blocks, BS)
        self.r = kvcache.BlockPool(num_blocks, BS)
        self.gt = torch.full((B, max_blocks), -1, dtype=torch.int32, device=DEV)
        self.rt = np.full((B, max_blocks), -1, np.int32)
        self.gs = torch.zeros(B, dtype=torch.int32, device=DEV)
        self.rs = np.zeros(B, np.int32)

    def t(self, a):
        return torch.tensor(np.asarray(a), dtype=torch.int32, device=DEV)

    def check(self):
        torch.cuda.synchronize()
        top = int(self.g.free_top.item())
        assert top == self.r.free_top
        np.testing.assert_array_equal(self.g.free_stack.cpu().numpy()[:top],
                                      self.r.free_stack[:top])
        np.testing.assert_array_equal(self.g.refcount.cpu().numpy()[:self.r.num_blocks],
                                      self.r.refcount)
        np.testing.assert_array_equal(self.gt.cpu().numpy(), self.rt)
        np.testing.assert_array_equal(self.gs.cpu().numpy(), self.rs)

    def reserve(self, k):
        self.g.reserve(self.gs, self.t(k), self.gt)
        self.r.reserve(self.rs, k, self.rt)

    def prefill(self, S):
        self.g.reserve(self.gs, self.t(np.asarray(S) - 1), self.gt)
        self.r.reserve(self.rs, np.asarray(S) - 1, self.rt)
        self.gs.copy_(self.t(S))
        self.rs[:] = S

    def admit(self, ids, n):
        """Give requests `ids` (empty rows) fresh blocks for [0, n) and seq_len n."""
        ids = np.asarray(ids)
        n = np.asarray(n)
        rows = torch.tensor(ids, device=DEV)
        gsub = self.gt[rows].contiguous()
        rsub = self.rt[ids].copy()
        self.g.reserve(torch.zeros(ids.size, dtype=torch.int32, device=DEV), self.t(n - 1), gsub)
        self.r.reserve(np.zeros(ids.size, np.int32), n - 1, rsub)
        self.gt[rows] = gsub
        self.rt[ids] = rsub
        self.gs[rows] = self.t(n)
        self.rs[ids] = n

    def commit(self, k, acc):
        nf = torch.full((len(acc),), -7, dtype=torch.int32, device=DEV)
        self.g.commit_rollback(self.t(k), self.t(acc), self.gs, self.gt, nf)
        want = self.r.commit_rollback(k, acc, self.rs, self.rt)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(nf.cpu().numpy(), want)

    def release(self, ids):
        nf = torch.full((len(ids),), -7, dtype=torch.int32, device=DEV)
        self.g.release(self.t(ids), self.gs, self.gt, nf)
        want = self.r.release(ids, self.rs, self.rt)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(nf.cpu().numpy(), want)


@pytest.mark.parametrize("B,BS", [(12, 16), (1500, 16), (64, 1)])
def test_random_cycles_bit_exact(ver, B, BS):
    rng = np.random.default_rng(B)
    mb = 700
    pr = Pair(ver, B * mb, BS, B, mb)
    pr.check()
    pr.prefill(rng.integers(1, 300 if BS == 1 else 8192, B))
    pr.check()
    for step in range(25):
        k = rng.integers(0, 9, B)
        pr.reserve(k)
        pr.check()
        acc = np.array([rng.integers(-1, kb + 1) for kb in k])
        pr.commit(k, acc)
        pr.check()
        if step % 8 == 7:
            ids = rng.choice(B, max(1, B // 5), replace=False)
            pr.release(ids)
            pr.check()
            pr.admit(ids, rng.integers(1, 200, ids.size))
            pr.check()
    assert ver.error() == 0


def test_oom_is_all_or_nothing(ver):
    pr = Pair(ver, 40, 16, 4, 16)
    pr.prefill([100, 100, 100, 100])                      # 4 x 7 = 28 blocks
    pr.check()
    before = (pr.g.free_stack.clone(), pr.g.free_top.clone(), pr.g.refcount.clone(), pr.gt.clone())
    pr.g.reserve(pr.gs, pr.t([60, 60, 60, 60]), pr.gt)   # needs 4 x 4 = 16 > 12 free
    torch.cuda.synchronize()
    assert ver.error() == binding.SV_ERR_OOM
    for a, b in zip(before, (pr.g.free_stack, pr.g.free_top, pr.g.refcount, pr.gt)):
        assert torch.equal(a, b)


def test_bad_accepted_is_refused(ver):
    pr = Pair(ver, 64, 16, 2, 8)
    pr.prefill([20, 5])
    pr.reserve([4, 4])
    pr.check()
    snap = (pr.gt.clone(), pr.gs.clone(), pr.g.refcount.clone())
    pr.g.commit_rollback(pr.t([4, 4]), pr.t([5, 1]), pr.gs, pr.gt)   # 5 > k
    torch.cuda.synchronize()
    assert ver.error() == binding.SV_ERR_STATE
    assert torch.equal(snap[0], pr.gt) and torch.equal(snap[1], pr.gs)
    assert torch.equal(snap[2], pr.g.refcount)


def test_shared_prefix_fork_cycles_and_release(ver):
    """Groups of 4 share a 1024-token prefix (64 blocks, refcount 4): rollback
    never touches a shared block; releasing members drops shared refs and frees
    them with the last member, in the reference order."""
    rng = np.random.default_rng(3)
    G, groups, BS = 4, 16, 16
    B = G * groups
    pr = Pair(ver, 64 * groups + B * 8 + 64, BS, B, 80)
    leaders = np.arange(0, B, G)
    pr.admit(leaders, np.full(leaders.size, 1024))       # 64 whole blocks each
    src = np.repeat(leaders, G - 1)
    dst = np.array([l + j for l in leaders for j in range(1, G)])
    pr.g.fork_prefix(pr.t(src), pr.t(dst), pr.t(np.full(dst.size, 64)), pr.gt)
    pr.r.fork_prefix(src, dst, np.full(dst.size, 64), pr.rt)
    pr.gs.fill_(1024)
    pr.rs[:] = 1024
    pr.check()
    assert (pr.r.refcount[pr.rt[leaders, :64]] == G).all()
    shared = pr.rt[:, :64].copy()
    for step in range(6):
        k = np.full(B, 4)
        pr.reserve(k)
        pr.commit(k, rng.integers(0, 5, B))
        pr.check()
        np.testing.assert_array_equal(pr.rt[:, :64], shared)
    assert (pr.r.refcount[np.unique(shared)] == G).all()
    pr.release(np.arange(1, B, 2))                        # two members of every group
    pr.check()
    pr.release(np.arange(0, B, 2))                        # the rest: shared blocks freed
    pr.check()
    assert pr.r.free_top == pr.r.num_blocks
    assert ver.error() == 0


def test_contiguous_rollback(ver):
    wp = torch.tensor([32, 7, 100], dtype=torch.int32, device=DEV)
    acc = torch.tensor([3, -1, 0], dtype=torch.int32, device=DEV)
    binding.kv_rollback_contig(ver.handle, acc, wp)
    ref = np.array([32, 7, 100])
    kvcache.rollback_contiguous([3, -1, 0], ref)
    assert wp.cpu().numpy().tolist() == ref.tolist()


def test_verify_then_commit_matches_no_speculation_recompute(ver):
    """The whole cycle on the GPU: reserve, the harness writes candidate K/V
    (the target pass), spec_verify, kv_commit_rollback; the valid cache equals
    a recompute of the committed history and the next-step distributions agree
    (forced rejections at the first/middle/last draft and at block edges)."""
    inp = W.paged_bf16(V=4096)
    B, k = inp["tokens"].shape
    BS, mb = 16, 160
    model = ToyAttention(seed=7)
    nblk = B * mb
    payload = PagedPayload(model, nblk, BS)
    pool = binding.BlockPool(ver.handle, nblk, BS)
    table = torch.full((B, mb), -1, dtype=torch.int32, device=DEV)
    seq = torch.zeros(B, dtype=torch.int32, device=DEV)
    S = inp["seq_len"].astype(np.int64)
    rng = np.random.default_rng(1)
    hist = [list(rng.integers(0, 4096, int(S[b]) + 1)) for b in range(B)]
    pool.reserve(seq, torch.tensor(S - 1, dtype=torch.int32, device=DEV), table)
    seq.copy_(torch.tensor(S, dtype=torch.int32))
    tbl = table.cpu().numpy()
    for b in range(B):
        payload.write(tbl[b], hist[b][:S[b]], list(range(S[b])))
    dev = device_io.to_device(inp, DEV)
    pool.reserve(seq, dev["k"], table)
    tbl = table.cpu().numpy()
    for b in range(B):                                    # the target pass writes candidates
        y = inp["tokens"][b, :k].tolist()
        payload.write(tbl[b], [hist[b][-1]] + y, list(range(S[b], S[b] + k + 1)))
    out = ver.verify(**dev)
    pool.commit_rollback(dev["k"], out["accepted"], seq, table)
    torch.cuda.synchronize()
    assert ver.error() == 0
    parity.compare(inp, out)
    acc = out["accepted"].cpu().numpy()
    tok = out["out_tokens"].cpu().numpy()
    seq_h, tbl = seq.cpu().numpy(), table.cpu().numpy()
    for b in range(B):
        a = int(acc[b])
        hist[b] = hist[b] + inp["tokens"][b, :a].tolist() + [int(tok[b, a])]
        assert seq_h[b] == len(hist[b]) - 1 == S[b] + 1 + a
        valid = payload.gather(tbl[b], int(seq_h[b]))
        recompute = model.kv(hist[b][:-1], list(range(len(hist[b]) - 1)))
        np.testing.assert_array_equal(valid, recompute)
        np.testing.assert_array_equal(
            model.next_distribution(valid, hist[b][-1], int(seq_h[b])),
            model.next_distribution(recompute, hist[b][-1], len(hist[b]) - 1))
        assert (tbl[b] >= 0).sum() == -(-int(seq_h[b]) // BS)
    assert (seq_h[4] % BS) == 0 and (seq_h[5] % BS) == 1   # block-edge scenarios


def test_draft_cache_realignment_bit_exact(ver):
    """Target and draft pools side by side: each round the draft catches up and
    proposes (its cache covers [0, S + k)), then kv_commit_draft realigns it
    with the committed history; GPU and reference agree bit for bit."""
    rng = np.random.default_rng(21)
    B, BS, mb = 48, 16, 700
    tgt = Pair(ver, B * mb, BS, B, mb)
    drf = Pair(ver, B * mb, BS, B, mb)
    S0 = rng.integers(1, 4000, B)
    tgt.prefill(S0)
    drf.prefill(S0)                                     # the draft saw the same prefix
    for step in range(20):
        k = rng.integers(1, 9, B)
        tgt.reserve(k)
        S = tgt.rs.copy()
        D = drf.rs.copy()
        extra = S + k - D                               # the draft processes D .. S + k - 1
        drf.reserve(extra - 1)
        drf.gs.copy_(drf.t(S + k))
        drf.rs[:] = S + k
        acc = np.array([rng.integers(-1, kb + 1) for kb in k])
        nf = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        drf.g.commit_draft(tgt.gs, drf.t(acc), drf.gs, drf.gt, nf)
        want = drf.r.commit_draft(tgt.rs, acc, drf.rs, drf.rt)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(nf.cpu().numpy(), want)
        drf.check()
        tgt.commit(k, acc)
        tgt.check()
        assert (drf.rs <= tgt.rs).all()
    # a bad accepted value changes nothing
    snap = (drf.gt.clone(), drf.gs.clone(), drf.g.refcount.clone(), drf.g.free_top.clone())
    bad = np.zeros(B, np.int64)
    bad[3] = -2
    drf.g.commit_draft(tgt.gs, drf.t(bad), drf.gs, drf.gt)
    torch.cuda.synchronize()
    assert ver.error() == binding.SV_ERR_STATE
    for a, b in zip(snap, (drf.gt, drf.gs, drf.g.refcount, drf.g.free_top)):
        assert torch.equal(a, b)


def test_copy_on_write_and_commit_by_copy_bit_exact(ver):
    """Paged payload [blocks, L, 2, H, BS, D] on both sides: requests fork
    prefixes whose last block is partial, reserve with copy-on-write, stage
    candidate K/V and commit the accepted entries by copy.  Pools, tables and
    the whole payload match the reference bit for bit every round."""
    rng = np.random.default_rng(31)
    B, BS, mb, L, H, D = 24, 16, 64, 2, 2, 8
    nblk = B * mb
    pr = Pair(ver, nblk, BS, B, mb)
    kv_r = rng.standard_normal((nblk, L, 2, H, BS, D)).astype(np.float32)
    kv_g = torch.tensor(kv_r, device=DEV)
    scratch = torch.empty(3 * B, dtype=torch.int32, device=DEV)
    # requests 0..7 get prefixes; 8..23 fork them (the last forked block is partial)
    pr.admit(np.arange(8), rng.integers(20, 300, 8))
    src = np.arange(8).repeat(2)
    dst = np.arange(8, 24)
    nblocks = np.array([kvcache.ceil_div(int(pr.rs[s]), BS) for s in src])
    pr.g.fork_prefix(pr.t(src), pr.t(dst), pr.t(nblocks), pr.gt)
    pr.r.fork_prefix(src, dst, nblocks, pr.rt)
    pr.gs[torch.tensor(dst, device=DEV)] = pr.t(pr.rs[src])
    pr.rs[dst] = pr.rs[src]
    pr.check()
    kmax = 6
    for step in range(8):
        k = rng.integers(0, kmax + 1, B)
        pr.g.reserve_cow(pr.gs, pr.t(k), pr.gt, kv_g, scratch)
        pr.r.reserve_cow(pr.rs, k, pr.rt, kv_r)
        pr.check()
        np.testing.assert_array_equal(kv_g.cpu().numpy(), kv_r)
        stage = rng.standard_normal((B, kmax + 1, L, 2, H, D)).astype(np.float32)
        acc = np.array([rng.integers(-1, kb + 1) for kb in k])
        binding.kv_commit_copy(ver.handle, pr.t(acc), pr.gs, pr.gt, BS, nblk,
                               torch.tensor(stage, device=DEV), kv_g)
        kvcache.commit_copy(stage, acc, pr.rs, pr.rt, kv_r, BS)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(kv_g.cpu().numpy(), kv_r)
        pr.commit(k, acc)
        pr.check()
    assert ver.error() == 0
