"""Reference paged-KV cache manager for the verification cycle (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources (page titles; paragraphs counted on the page):
  [KV]  "Walk through KV-cache updates when speculative decoding rejects some
        draft tokens": candidate K/V is appended provisionally during the
        verify pass; after the first rejection the rejected positions are
        removed -- free the pages on a paged cache, rewind the write pointer on
        a contiguous one -- so the cache holds exactly the committed sequence.
  [RJ]  "Rejected speculative tokens remain in KV" (interview question),
        paragraphs 1-2: allocation is not acceptance; a physical block may stay
        allocated with only part of it valid if attention cannot read the rest.
  [CV]  "Keep cache validity aligned with the committed token history",
        paragraphs 1-4: the pending-token convention (cache length = processed
        tokens, the newest emitted token is pending), keep prefix plus the
        accepted proposals and leave the correction pending; block tables,
        ownership and reference counts decide which memory is valid; rollback of
        one request must not mutate another request's committed prefix.

State (all plain arrays, mirrored bit for bit by the CUDA path):
  free_stack [num_blocks] int32, free_top, refcount [num_blocks] int32,
  block_table [B][max_blocks] int32 (-1 = no block), seq_len [B] int32.

Readings:
  * seq_len S_b counts processed tokens; the pending token sits at position
    S_b.  The verify pass processes positions S_b .. S_b + k_b, so it needs
    blocks covering [0, S_b + k_b + 1).
  * after a pass with a_b accepted drafts: seq_len <- S_b + 1 + a_b (the old
    pending token and the accepted drafts are now processed; the correction or
    bonus token is the new pending token).  a_b = -1 (bad input) keeps S_b.
  * blocks j in [ceil(new/BS), ceil((S_b + k_b + 1)/BS)) are dropped: table
    entry cleared, refcount decremented, pushed on the free stack when it
    reaches 0.  A block with at least one valid slot is kept.
  * order: requests ascending, j ascending, for pops and pushes alike; the
    free stack starts as [n-1, ..., 1, 0] so that blocks pop as 0, 1, 2, ...
  * a fork shares whole blocks (a partially filled last block included);
    reserve refuses to append into a partially filled block whose refcount is
    above 1, reserve_cow copies it first (copy-on-write).
  * a draft model's cache keeps min(D_b, committed length) of its own
    processed positions (see commit_draft).
"""

from __future__ import annotations

import numpy as np


class CacheError(Exception):
    pass


class OutOfBlocks(CacheError):
    pass


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class BlockPool:
    """Free list + refcounts of a pool of num_blocks blocks of block_size slots."""

    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.free_stack = np.arange(self.num_blocks - 1, -1, -1, dtype=np.int32)
        self.free_top = self.num_blocks
        self.refcount = np.zeros(self.num_blocks, np.int32)

    def copy(self) -> "BlockPool":
        c = BlockPool.__new__(BlockPool)
        c.num_blocks, c.block_size = self.num_blocks, self.block_size
        c.free_stack = self.free_stack.copy()
        c.free_top = self.free_top
        c.refcount = self.refcount.copy()
        return c

    def _pop(self) -> int:
        self.free_top -= 1
        blk = int(self.free_stack[self.free_top])
        self.refcount[blk] = 1
        return blk

    def _drop(self, blk: int) -> bool:
        """Decrement blk's refcount; push it on the free stack if it hit 0."""
        if not (0 <= blk < self.num_blocks) or self.refcount[blk] <= 0:
            raise CacheError(f"drop of unowned block {blk}")
        self.refcount[blk] -= 1
        if self.refcount[blk] == 0:
            self.free_stack[self.free_top] = blk
            self.free_top += 1
            return True
        return False

    # ------------------------------------------------------------------ #
    def reserve(self, seq_len, k, block_table) -> None:
        """Lookahead allocation before the verify pass ([RJ] paragraph 1).

        Covers positions [0, S_b + k_b + 1) for every request; all-or-nothing.
        """
        BS = self.block_size
        B = len(seq_len)
        need = []
        for b in range(B):
            S, kb = int(seq_len[b]), int(k[b])
            have, want = ceil_div(S, BS), ceil_div(S + kb + 1, BS)
            if S < 0 or kb < 0 or want > block_table.shape[1]:
                raise CacheError(f"request {b}: bad sizes")
            row = block_table[b]
            if (row[:have] < 0).any() or (row[have:want] >= 0).any():
                raise CacheError(f"request {b}: table does not match seq_len")
            if S % BS and self.refcount[row[have - 1]] > 1:
                raise CacheError(f"request {b}: append into a shared partial block")
            need.append(want - have)
        if sum(need) > self.free_top:
            raise OutOfBlocks(f"need {sum(need)} blocks, {self.free_top} free")
        for b in range(B):
            have = ceil_div(int(seq_len[b]), BS)
            for t in range(need[b]):
                block_table[b, have + t] = self._pop()

    def reserve_cow(self, seq_len, k, block_table, kv) -> None:
        """Lookahead allocation with copy-on-write of a shared partial block
        ([CV] paragraph 4: copy-on-write addresses physical sharing while the
        decoder keeps the token and position mapping).

        Like reserve, but a request whose last held block is partially filled
        (r = S_b % BS > 0) and shared (refcount > 1 when the call starts) first
        gets a fresh block holding a copy of that block's valid slots [0, r)
        for every layer, K/V and head; the table entry points at the copy and
        the shared block loses one reference per copy, staying unchanged with
        its other owners.  Pops run in (request, j) order, the copy taking
        index j = have - 1; a shared block left without references (all its
        owners copied) is pushed on the free stack after every pop, in request
        order.  All or nothing.  kv: payload [num_blocks, L, 2, H, BS, D].
        """
        BS = self.block_size
        B = len(seq_len)
        need, cow = [], []
        for b in range(B):
            S, kb = int(seq_len[b]), int(k[b])
            have, want = ceil_div(S, BS), ceil_div(S + kb + 1, BS)
            if S < 0 or kb < 0 or want > block_table.shape[1]:
                raise CacheError(f"request {b}: bad sizes")
            row = block_table[b]
            if (row[:have] < 0).any() or (row[have:want] >= 0).any():
                raise CacheError(f"request {b}: table does not match seq_len")
            c = bool(S % BS) and self.refcount[row[have - 1]] > 1
            need.append(want - have + int(c))
            cow.append(c)
        if sum(need) > self.free_top:
            raise OutOfBlocks(f"need {sum(need)} blocks, {self.free_top} free")
        dropped = []
        for b in range(B):
            S = int(seq_len[b])
            have = ceil_div(S, BS)
            row = block_table[b]
            if cow[b]:
                old, new, r = int(row[have - 1]), self._pop(), S % BS
                kv[new, :, :, :, :r, :] = kv[old, :, :, :, :r, :]
                dropped.append(old)
                row[have - 1] = new
            for t in range(need[b] - int(cow[b])):
                row[have + t] = self._pop()
        for old in dropped:  # after every pop: a freed block is not reused in this call
            self._drop(old)

    def commit_rollback(self, k, accepted, seq_len, block_table):
        """Commit the accepted prefix, roll back the rejected tail ([KV], [CV] 2-3).

        Returns n_freed [B] (blocks pushed on the free stack per request).
        """
        BS = self.block_size
        B = len(seq_len)
        n_freed = np.zeros(B, np.int32)
        for b in range(B):
            S, kb, a = int(seq_len[b]), int(k[b]), int(accepted[b])
            if not (-1 <= a <= kb):
                raise CacheError(f"request {b}: accepted {a} outside [-1, {kb}]")
            new = S if a < 0 else S + 1 + a
            for j in range(ceil_div(new, BS), ceil_div(S + kb + 1, BS)):
                blk = int(block_table[b, j])
                block_table[b, j] = -1
                n_freed[b] += self._drop(blk)
            seq_len[b] = new
        return n_freed

    def commit_draft(self, seq_len, accepted, draft_len, block_table):
        """Realign a draft model's cache with the committed history ([SD]
        section 4, "update cache state": the draft cache is reconciled with the
        corrected token; [CV] paragraph 4: the draft follows its own processed-
        state convention and is never filled from target K/V).

        Reading: the draft's cache holds draft_len[b] = D_b processed positions
        (however far its own proposal loop went).  After the pass the committed
        history has S_b + 1 + a_b processed tokens (S_b when a_b = -1), so the
        draft keeps min(D_b, that) positions; a shorter draft catches up on the
        committed tokens next round.  Blocks j in [ceil(keep/BS), ceil(D_b/BS))
        are dropped in (request, j) order.  seq_len is the TARGET length before
        the pass (S_b).  Returns n_freed [B].
        """
        BS = self.block_size
        B = len(draft_len)
        n_freed = np.zeros(B, np.int32)
        for b in range(B):
            S, a, D = int(seq_len[b]), int(accepted[b]), int(draft_len[b])
            if S < 0 or D < 0 or a < -1 or ceil_div(D, BS) > block_table.shape[1]:
                raise CacheError(f"request {b}: bad sizes")
            if (block_table[b, :ceil_div(D, BS)] < 0).any():
                raise CacheError(f"request {b}: draft table does not cover its length")
            keep = min(D, S if a < 0 else S + 1 + a)
            for j in range(ceil_div(keep, BS), ceil_div(D, BS)):
                blk = int(block_table[b, j])
                block_table[b, j] = -1
                n_freed[b] += self._drop(blk)
            draft_len[b] = keep
        return n_freed

    def fork_prefix(self, src, dst, n_blocks, block_table) -> None:
        """Share the first n whole blocks of request src with request dst ([CV] 4)."""
        for s, d, n in zip(src, dst, n_blocks):
            if (block_table[d, :n] >= 0).any() or (block_table[s, :n] < 0).any():
                raise CacheError(f"fork {s}->{d}: bad tables")
            for j in range(int(n)):
                blk = int(block_table[s, j])
                block_table[d, j] = blk
                self.refcount[blk] += 1

    def release(self, req_ids, seq_len, block_table):
        """Drop every block a finished request holds; shared blocks just lose a ref."""
        n_freed = np.zeros(len(req_ids), np.int32)
        for i, b in enumerate(req_ids):
            row = block_table[b]
            for j in range(row.shape[0]):
                if row[j] < 0:
                    break
                blk = int(row[j])
                row[j] = -1
                n_freed[i] += self._drop(blk)
            seq_len[b] = 0
        return n_freed


def commit_copy(stage, accepted, seq_len, block_table, kv, block_size, path=None) -> None:
    """Commit by copy ([KV]: candidate K/V is written provisionally and only the
    accepted part is kept; [RJ] paragraph 1: allocation is not acceptance).

    The verify pass wrote the K/V of positions S_b .. S_b + k_b (the pending
    token and the drafts) into stage [B, kmax + 1, L, 2, H, D]; this copies
    entries i = 0 .. a_b (positions S_b .. S_b + a_b) into their paged slots
    kv[table[b, p // BS], :, :, :, p % BS, :]; a_b = -1 copies nothing, and
    rejected entries are never written.  seq_len: S_b, the length before
    commit_rollback updates it.

    Token tree ([CV] paragraph 3: gather the accepted path into the cache
    layout): stage holds one entry per tree node (entry 0 the pending token)
    and path[b][i - 1] names the node whose entry goes to position S_b + i.
    Entries of nodes off the path (siblings of the accepted branch and their
    descendants) are never written, so no cache position refers to them.
    """
    for b in range(len(accepted)):
        S, a = int(seq_len[b]), int(accepted[b])
        for i in range(a + 1):
            p = S + i
            blk = int(block_table[b, p // block_size])
            if blk < 0:
                raise CacheError(f"request {b}: position {p} has no block")
            e = i if path is None or i == 0 else int(path[b][i - 1])
            kv[blk, :, :, :, p % block_size, :] = stage[b, e]


def rollback_contiguous(accepted, write_ptr) -> None:
    """Contiguous cache: rewind the write pointer to S_b + 1 + a_b ([KV])."""
    for b in range(len(write_ptr)):
        a = int(accepted[b])
        if a >= 0:
            write_ptr[b] = int(write_ptr[b]) + 1 + a
