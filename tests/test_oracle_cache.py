"""Pins of the reference cache manager: a hand-derived scenario, brute-force
recounts of ownership, forced-rejection rounds checked through a toy attention
model against a no-speculation recompute, and shared-prefix isolation."""

import numpy as np
import pytest

from oracle.kvcache import (BlockPool, CacheError, OutOfBlocks, ceil_div, commit_copy,
                            rollback_contiguous)
from tests.toy_model import PagedPayload, ToyAttention


def _check_invariants(pool: BlockPool, table, seq_len=None):
    """Brute-force recount: refcount == table references; free set == unreferenced."""
    refs = np.zeros(pool.num_blocks, np.int64)
    for row in table:
        live = row[row >= 0]
        n = live.size
        assert (row[:n] >= 0).all() and (row[n:] < 0).all(), "table rows must be prefixes"
        np.add.at(refs, live, 1)
    np.testing.assert_array_equal(refs, pool.refcount)
    free = pool.free_stack[:pool.free_top]
    assert len(set(free.tolist())) == free.size
    assert set(free.tolist()) == set(np.flatnonzero(refs == 0).tolist())
    assert pool.free_top + (refs > 0).sum() == pool.num_blocks
    if seq_len is not None:
        for b, S in enumerate(seq_len):
            assert (table[b] >= 0).sum() >= ceil_div(int(S), pool.block_size)


def test_hand_derived_scenario():
    pool = BlockPool(6, 4)
    np.testing.assert_array_equal(pool.free_stack, [5, 4, 3, 2, 1, 0])
    table = np.full((3, 6), -1, np.int32)
    seq = np.array([0, 0, 0], np.int32)
    pool.reserve(seq[:2], [4, 6], table)                 # covers [0,5) and [0,7)
    np.testing.assert_array_equal(table[:2], [[0, 1, -1, -1, -1, -1], [2, 3, -1, -1, -1, -1]])
    assert pool.free_top == 2
    freed = pool.commit_rollback([4, 6], [1, 6], seq[:2], table)
    np.testing.assert_array_equal(seq[:2], [2, 7])
    np.testing.assert_array_equal(freed, [1, 0])
    assert pool.free_top == 3 and pool.free_stack[2] == 1
    np.testing.assert_array_equal(pool.refcount, [1, 0, 1, 1, 0, 0])
    pool.reserve(seq[:2], [3, 3], table)
    np.testing.assert_array_equal(table[:2], [[0, 1, -1, -1, -1, -1], [2, 3, 4, -1, -1, -1]])
    pool.commit_rollback([3, 3], [0, 3], seq[:2], table)
    np.testing.assert_array_equal(seq[:2], [3, 11])
    assert pool.free_top == 2
    np.testing.assert_array_equal(pool.free_stack[:2], [5, 1])
    np.testing.assert_array_equal(pool.refcount, [1, 0, 1, 1, 1, 0])
    before = (pool.free_stack.copy(), pool.free_top, pool.refcount.copy(), table.copy())
    with pytest.raises(OutOfBlocks):                      # needs 2 + 2 > 2 free
        pool.reserve(seq[:2], [8, 8], table)
    np.testing.assert_array_equal(pool.free_stack, before[0])
    assert pool.free_top == before[1]
    np.testing.assert_array_equal(table, before[3])
    # fork one whole block of request 1 into request 2, then release both
    pool.fork_prefix([1], [2], [1], table)
    assert pool.refcount[2] == 2 and table[2, 0] == 2
    pool.release([1], seq, table)
    np.testing.assert_array_equal(pool.free_stack[:pool.free_top], [5, 1, 3, 4])
    assert pool.refcount[2] == 1
    pool.release([2], seq, table)
    np.testing.assert_array_equal(pool.free_stack[:pool.free_top], [5, 1, 3, 4, 2])
    _check_invariants(pool, table)


def test_bad_accepted_and_shared_partial_append_are_refused():
    pool = BlockPool(8, 4)
    table = np.full((2, 4), -1, np.int32)
    seq = np.array([0, 0], np.int32)
    pool.reserve(seq, [5, 0], table)
    with pytest.raises(CacheError):                        # accepted > k
        pool.commit_rollback([5, 0], [6, 0], seq.copy(), table.copy())
    with pytest.raises(CacheError):                        # fork onto an owned slot
        pool.copy().fork_prefix([0], [1], [2], table.copy())
    pool.commit_rollback([5, 0], [4, 0], seq, table)       # seq -> [5, 1]
    np.testing.assert_array_equal(seq, [5, 1])
    shared = pool.copy()
    shared.refcount[table[0, 1]] += 1                      # block 1 of request 0 is partial
    with pytest.raises(CacheError):
        shared.reserve(seq, [1, 0], table.copy())


def test_random_cycles_keep_ownership_consistent():
    rng = np.random.default_rng(0)
    BS, B = 16, 12
    pool = BlockPool(400, BS)
    table = np.full((B, 64), -1, np.int32)
    seq = np.zeros(B, np.int32)
    pre = rng.integers(1, 300, B)
    pool.reserve(seq, pre - 1, table)                      # prefill [0, pre)
    seq[:] = pre
    _check_invariants(pool, table, seq)
    for step in range(40):
        k = rng.integers(0, 9, B)
        pool.reserve(seq, k, table)
        acc = np.array([rng.integers(-1, kb + 1) for kb in k])
        pool.commit_rollback(k, acc, seq, table)
        _check_invariants(pool, table, seq)
        for b in range(B):
            assert (table[b] >= 0).sum() == ceil_div(int(seq[b]), BS)
        if step % 10 == 9:
            gone = rng.choice(B, 3, replace=False)
            pool.release(gone, seq, table)
            _check_invariants(pool, table)
            for b in gone:
                n = int(rng.integers(1, 200))
                pool.reserve(np.array([0]), [n - 1], table[b:b + 1])
                seq[b] = n
            _check_invariants(pool, table, seq)


@pytest.mark.parametrize("reject_at", [0, 2, 4, None])
@pytest.mark.parametrize("block_edge", [False, True])
def test_rollback_matches_no_speculation_recompute(reject_at, block_edge):
    """Forced rejection at the first / middle / last draft (None: all accepted,
    bonus kept pending), optionally placed so the kept prefix ends on a block
    boundary: the valid cache equals a recompute of the committed history and
    the next-step distribution agrees."""
    BS, k = 16, 5
    m = ToyAttention(seed=1)
    rng = np.random.default_rng(2)
    pool = BlockPool(64, BS)
    payload = PagedPayload(m, 64, BS)
    table = np.full((1, 16), -1, np.int32)
    S = 37
    a = k if reject_at is None else reject_at
    if block_edge:
        S = 48 - 1 - a                                 # kept length S + 1 + a = 48
    history = list(rng.integers(0, 1000, S + 1))       # S processed + 1 pending
    seq = np.array([0], np.int32)
    pool.reserve(seq, [S - 1], table)                  # prefill positions [0, S)
    payload.write(table[0], history[:S], list(range(S)))
    seq[0] = S
    for rnd in range(3):
        drafts = list(rng.integers(0, 1000, k))
        pool.reserve(seq, [k], table)
        S0 = int(seq[0])
        # the verify pass writes K/V for [pending, y_1..y_k] at S0 .. S0 + k
        payload.write(table[0], [history[-1]] + drafts, list(range(S0, S0 + k + 1)))
        aa = a if rnd == 0 else int(rng.integers(0, k + 1))
        corr = int(rng.integers(0, 1000))
        pool.commit_rollback([k], [aa], seq, table)
        history = history + drafts[:aa] + [corr]
        assert seq[0] == S0 + 1 + aa == len(history) - 1
        valid = payload.gather(table[0], int(seq[0]))
        recompute = m.kv(history[:-1], list(range(len(history) - 1)))
        np.testing.assert_array_equal(valid, recompute)
        got = m.next_distribution(valid, history[-1], int(seq[0]))
        want = m.next_distribution(recompute, history[-1], len(history) - 1)
        np.testing.assert_array_equal(got, want)
        _check_invariants(pool, table, seq)
        if block_edge and rnd == 0:
            assert (table[0] >= 0).sum() == 48 // BS   # no partially empty block kept


def test_shared_prefix_is_never_mutated_by_rollback():
    BS, G, k = 16, 4, 4
    m = ToyAttention(seed=3)
    rng = np.random.default_rng(4)
    pool = BlockPool(200, BS)
    payload = PagedPayload(m, 200, BS)
    table = np.full((G, 32), -1, np.int32)
    seq = np.zeros(G, np.int32)
    prefix = 64                                          # 4 whole blocks
    hist0 = list(rng.integers(0, 500, prefix))
    pool.reserve(seq[:1], [prefix - 1], table[:1])
    payload.write(table[0], hist0, list(range(prefix)))
    pool.fork_prefix([0] * (G - 1), list(range(1, G)), [prefix // BS] * (G - 1), table)
    shared = table[0, :prefix // BS].copy()
    np.testing.assert_array_equal(pool.refcount[shared], G)
    snap = payload.data[shared].copy()
    seq[:] = prefix
    hist = [hist0 + [int(rng.integers(0, 500))] for _ in range(G)]
    for rnd in range(6):
        pool.reserve(seq, [k] * G, table)
        for b in range(G):
            S0 = int(seq[b])
            drafts = list(rng.integers(0, 500, k))
            payload.write(table[b], [hist[b][-1]] + drafts, list(range(S0, S0 + k + 1)))
            hist[b] = hist[b] + drafts
        acc = rng.integers(0, k + 1, G)
        pool.commit_rollback([k] * G, acc, seq, table)
        for b in range(G):
            S0 = len(hist[b]) - k - 1
            hist[b] = hist[b][:S0 + 1 + acc[b]] + [int(rng.integers(0, 500))]
            assert seq[b] == len(hist[b]) - 1
            np.testing.assert_array_equal(payload.gather(table[b], int(seq[b])),
                                          m.kv(hist[b][:-1], list(range(len(hist[b]) - 1))))
        np.testing.assert_array_equal(table[:, :prefix // BS], np.tile(shared, (G, 1)))
        np.testing.assert_array_equal(payload.data[shared], snap)
        np.testing.assert_array_equal(pool.refcount[shared], G)
        _check_invariants(pool, table, seq)
    pool.release([1, 2], seq, table)
    np.testing.assert_array_equal(pool.refcount[shared], G - 2)
    pool.release([0, 3], seq, table)
    assert pool.free_top == pool.num_blocks
    _check_invariants(pool, table)


def test_contiguous_write_pointer_rollback():
    m = ToyAttention(seed=5)
    rng = np.random.default_rng(6)
    k, S = 5, 32
    buf = np.zeros((64, m.L, 2, m.H, m.d), np.float32)
    history = list(rng.integers(0, 1000, S + 1))
    buf[:S] = m.kv(history[:S], list(range(S)))
    wp = np.array([S], np.int32)
    for a in (0, 3, 5, -1):
        S0 = int(wp[0])
        drafts = list(rng.integers(0, 1000, k))
        buf[S0:S0 + k + 1] = m.kv([history[-1]] + drafts, list(range(S0, S0 + k + 1)))
        rollback_contiguous([a], wp)
        if a >= 0:
            history = history + drafts[:a] + [int(rng.integers(0, 1000))]
        assert wp[0] == len(history) - 1
        np.testing.assert_array_equal(buf[:wp[0]], m.kv(history[:-1], list(range(wp[0]))))


# --------------------------------------------------------------------------- #
# draft-cache realignment
# --------------------------------------------------------------------------- #
def test_draft_commit_hand_scenario():
    """BS = 4, target length S = 5, k = 4 proposals; the draft processed the
    pending token and y_0..y_2 while proposing (D = S + k = 9, blocks 0-2)."""
    for a, keep, freed in [(1, 7, 1), (4, 9, 0), (-1, 5, 1), (3, 9, 0), (0, 6, 1)]:
        pool = BlockPool(6, 4)
        table = np.full((1, 4), -1, np.int32)
        pool.reserve(np.array([0]), [8], table)          # covers [0, 9)
        np.testing.assert_array_equal(table[0], [0, 1, 2, -1])
        D = np.array([9], np.int32)
        n = pool.commit_draft(np.array([5]), np.array([a]), D, table)
        assert D[0] == keep and n[0] == freed, (a, D, n)
        assert (table[0] >= 0).sum() == ceil_div(keep, 4)
        _check_invariants(pool, table)
    # a draft that processed everything (D = S + k + 1 = 10) keeps S + 1 + a
    pool = BlockPool(6, 4)
    table = np.full((1, 4), -1, np.int32)
    pool.reserve(np.array([0]), [9], table)
    D = np.array([10], np.int32)
    pool.commit_draft(np.array([5]), np.array([4]), D, table)
    assert D[0] == 10 and (table[0] >= 0).sum() == 3
    with pytest.raises(CacheError):                      # accepted below -1
        pool.copy().commit_draft(np.array([5]), np.array([-2]), D.copy(), table.copy())
    with pytest.raises(CacheError):                      # table shorter than the length
        pool.copy().commit_draft(np.array([5]), np.array([1]), np.array([13]), table.copy())


@pytest.mark.parametrize("reject_at", [0, 2, 4, None])
def test_draft_cache_matches_recompute_after_realignment(reject_at):
    """A toy draft proposes k tokens autoregressively into its own paged cache;
    after the draft commit its valid cache equals a recompute of the committed
    history, and after catching up on the committed tokens it has not processed
    its next-step distribution equals the recompute's."""
    BS, k = 8, 5
    draft = ToyAttention(seed=11)
    rng = np.random.default_rng(12)
    pool = BlockPool(64, BS)
    payload = PagedPayload(draft, 64, BS)
    table = np.full((1, 16), -1, np.int32)
    S = 21
    history = list(rng.integers(0, 1000, S + 1))          # S processed + 1 pending
    D = np.array([0], np.int32)
    pool.reserve(D, [S - 1], table)
    payload.write(table[0], history[:S], list(range(S)))
    D[0] = S
    for rnd in range(3):
        S0 = len(history) - 1                              # target length before the pass
        need = S0 + k - int(D[0])                           # the draft catches up, then proposes
        pool.reserve(D, [need - 1], table)
        todo = history[int(D[0]):] + []                    # committed tokens not yet processed
        drafts = list(rng.integers(0, 1000, k))
        seq_in = todo + drafts[:-1]                        # the draft processes up to y_{k-2}
        payload.write(table[0], seq_in, list(range(int(D[0]), int(D[0]) + len(seq_in))))
        D[0] = S0 + k
        a = (reject_at if reject_at is not None else k) if rnd == 0 else int(rng.integers(-1, k + 1))
        corr = int(rng.integers(0, 1000))
        pool.commit_draft(np.array([S0]), np.array([a]), D, table)
        history = history + (drafts[:a] + [corr] if a >= 0 else [])
        committed = S0 if a < 0 else S0 + 1 + a
        assert D[0] == min(S0 + k, committed)
        valid = payload.gather(table[0], int(D[0]))
        recompute = draft.kv(history[:int(D[0])], list(range(int(D[0]))))
        np.testing.assert_array_equal(valid, recompute)
        # catch up on committed-but-unprocessed tokens, then compare the next step
        n_proc = len(history) - 1
        cache = np.concatenate([valid, draft.kv(history[int(D[0]):n_proc], list(range(int(D[0]), n_proc)))])
        got = draft.next_distribution(cache, history[-1], n_proc)
        want = draft.next_distribution(draft.kv(history[:n_proc], list(range(n_proc))), history[-1], n_proc)
        np.testing.assert_array_equal(got, want)
        _check_invariants(pool, table)


# --------------------------------------------------------------------------- #
# commit by copy and copy-on-write
# --------------------------------------------------------------------------- #
def _gather(kv, row, n, BS):
    return np.stack([kv[row[j // BS], :, :, :, j % BS, :] for j in range(n)]) if n else \
        np.zeros((0,) + kv.shape[1:4] + kv.shape[5:], kv.dtype)


@pytest.mark.parametrize("reject_at", [0, 2, 4, None])
def test_commit_by_copy_matches_recompute(reject_at):
    """The verify pass writes candidate K/V to a staging buffer only; commit by
    copy moves the accepted entries into the paged cache, which then equals a
    recompute of the committed history (rejected entries never reach it)."""
    BS, k = 16, 5
    m = ToyAttention(seed=5)
    rng = np.random.default_rng(6)
    pool = BlockPool(32, BS)
    kv = np.full((32, m.L, 2, m.H, BS, m.d), np.nan, np.float32)   # unwritten slots are NaN
    table = np.full((1, 16), -1, np.int32)
    S = 30
    history = list(rng.integers(0, 1000, S + 1))
    seq = np.array([0], np.int32)
    pool.reserve(seq, [S - 1], table)
    stage0 = m.kv(history[:S], list(range(S)))
    for j in range(S):
        kv[table[0, j // BS], :, :, :, j % BS, :] = stage0[j]
    seq[0] = S
    for rnd in range(3):
        drafts = list(rng.integers(0, 1000, k))
        pool.reserve(seq, [k], table)
        S0 = int(seq[0])
        stage = m.kv([history[-1]] + drafts, list(range(S0, S0 + k + 1)))[None]
        a = (k if reject_at is None else reject_at) if rnd == 0 else int(rng.integers(0, k + 1))
        commit_copy(stage, [a], seq.copy(), table, kv, BS)
        pool.commit_rollback([k], [a], seq, table)
        history = history + drafts[:a] + [int(rng.integers(0, 1000))]
        n = int(seq[0])
        np.testing.assert_array_equal(_gather(kv, table[0], n, BS),
                                      m.kv(history[:-1], list(range(n))))
        _check_invariants(pool, table, seq)


def test_copy_on_write_keeps_forked_prefixes_isolated():
    """Three requests share a 37-token prefix (its third block is partial).
    Each appends its own drafts through reserve_cow; the shared partial block
    is copied before any write, every request's cache equals a recompute of its
    own history, and the blocks still shared are never written."""
    BS, k, S = 16, 4, 37
    m = ToyAttention(seed=7)
    rng = np.random.default_rng(8)
    pool = BlockPool(64, BS)
    kv = np.full((64, m.L, 2, m.H, BS, m.d), np.nan, np.float32)
    table = np.full((3, 16), -1, np.int32)
    prefix = list(rng.integers(0, 1000, S + 1))
    seq = np.array([0, 0, 0], np.int32)
    pool.reserve(seq[:1], [S - 1], table[:1])
    rows = m.kv(prefix[:S], list(range(S)))
    for j in range(S):
        kv[table[0, j // BS], :, :, :, j % BS, :] = rows[j]
    pool.fork_prefix([0, 0], [1, 2], [3, 3], table)
    seq[:] = S
    full_blocks = table[0, :2].copy()
    shared_full = kv[full_blocks].copy()
    partial = int(table[0, 2])
    partial_before = kv[partial].copy()
    hist = [list(prefix), list(prefix), list(prefix)]
    with pytest.raises(CacheError):                       # plain reserve refuses the append
        pool.copy().reserve(seq, [k, k, k], table.copy())
    for rnd in range(3):
        pool.reserve_cow(seq, [k, k, k], table, kv)
        if rnd == 0:
            # all three owners append in this call: each gets a copy (popped in
            # request order) and the original partial block returns to the free list
            assert partial not in {int(table[b, 2]) for b in range(3)}
            assert len({int(table[b, 2]) for b in range(3)}) == 3
            assert pool.refcount[partial] == 0 and partial in pool.free_stack[:pool.free_top]
            for b in range(3):
                np.testing.assert_array_equal(kv[table[b, 2], :, :, :, :S % BS],
                                              partial_before[:, :, :, :S % BS])
        drafts = [list(rng.integers(0, 1000, k)) for _ in range(3)]
        stage = np.stack([m.kv([hist[b][-1]] + drafts[b], list(range(int(seq[b]), int(seq[b]) + k + 1)))
                          for b in range(3)])
        acc = [int(rng.integers(0, k + 1)) for _ in range(3)]
        commit_copy(stage, acc, seq.copy(), table, kv, BS)
        pool.commit_rollback([k, k, k], acc, seq, table)
        for b in range(3):
            hist[b] = hist[b] + drafts[b][:acc[b]] + [int(rng.integers(0, 1000))]
            n = int(seq[b])
            assert n == len(hist[b]) - 1
            np.testing.assert_array_equal(_gather(kv, table[b], n, BS),
                                          m.kv(hist[b][:-1], list(range(n))))
        _check_invariants(pool, table, seq)
    np.testing.assert_array_equal(kv[full_blocks], shared_full)   # whole shared blocks untouched
    # an owner outside the call keeps the original block; the caller that appends copies it
    pool2 = BlockPool(16, BS)
    kv2 = np.zeros((16, 1, 2, 1, BS, 2), np.float32)
    t2 = np.full((2, 4), -1, np.int32)
    s2 = np.array([0, 0], np.int32)
    pool2.reserve(s2[:1], [S - 1], t2[:1])
    kv2[t2[0, 2], :, :, :, :S % BS] = 7.0
    pool2.fork_prefix([0], [1], [3], t2)
    s2[:] = S
    pool2.reserve_cow(s2[1:], [k], t2[1:], kv2)
    assert t2[0, 2] == 2 and t2[1, 2] != 2 and pool2.refcount[2] == 1
    np.testing.assert_array_equal(kv2[t2[1, 2], :, :, :, :S % BS], 7.0)
    _check_invariants(pool2, t2)


@pytest.mark.parametrize("forced_path", [[1, 3], [2, 4, 5], [2], []])
def test_tree_commit_gathers_the_accepted_branch(forced_path):
    """A token tree's candidate K/V sits in a staging buffer in node order; the
    accepted path (a branch switch when it starts at the second root child) is
    gathered into positions S..S+a and the cache equals a recompute of the
    committed history; no entry of a node off the path reaches the cache."""
    BS = 16
    m = ToyAttention(seed=11)
    rng = np.random.default_rng(12)
    pool = BlockPool(32, BS)
    kv = np.full((32, m.L, 2, m.H, BS, m.d), np.nan, np.float32)
    table = np.full((1, 16), -1, np.int32)
    S = 29
    history = list(rng.integers(0, 1000, S + 1))
    seq = np.array([0], np.int32)
    pool.reserve(seq, [S - 1], table)
    stage0 = m.kv(history[:S], list(range(S)))
    for j in range(S):
        kv[table[0, j // BS], :, :, :, j % BS, :] = stage0[j]
    seq[0] = S
    # nodes 1, 2 under the root; 3 under 1; 4 under 2; 5 under 4
    parent = [0, 0, 1, 2, 4]
    depth = [0, 1, 1, 2, 2, 3]
    toks = list(rng.integers(0, 1000, 5))
    for i in range(1, len(forced_path)):
        assert parent[forced_path[i] - 1] == forced_path[i - 1]
    dmax = max(depth)
    pool.reserve(seq, [dmax], table)
    stage = m.kv([history[-1]] + toks, [S + d for d in depth])[None]
    # nodes off the path get poisoned entries: any leak shows up as a mismatch
    off = [j for j in range(1, 6) if j not in forced_path]
    stage[0, off] = np.float32(1e30)
    a = len(forced_path)
    commit_copy(stage, [a], seq.copy(), table, kv, BS, path=[forced_path])
    pool.commit_rollback([dmax], [a], seq, table)
    committed = history + [toks[j - 1] for j in forced_path]
    n = int(seq[0])
    assert n == S + 1 + a
    np.testing.assert_array_equal(_gather(kv, table[0], n, BS),
                                  m.kv(committed, list(range(n))))
    _check_invariants(pool, table, seq)
