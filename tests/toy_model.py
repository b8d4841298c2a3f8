"""A synthetic toy attention "target model" for cache-state tests.

The pages' rollback tests compare the target's next-step distribution after a
speculative round with a recompute that never speculated ("Rejected speculative
tokens remain in KV", paragraph 3; "Keep cache validity aligned with the
committed token history", paragraph 5).  No trained weights exist here, so this
deterministic toy model stands in: for token t at absolute position j and each
layer/head, K_j = e(t) Wk + r(j), V_j = e(t) Wv + r'(j); the next-step logits
are Wo . sum_j softmax(q . K_j / sqrt(d)) V_j over the valid positions plus the
pending token itself.  Embeddings are closed-form in t, so any vocabulary works.
"""

from __future__ import annotations

import numpy as np


class ToyAttention:
    def __init__(self, layers=2, heads=4, head_dim=16, out_vocab=64, seed=0):
        rng = np.random.default_rng(seed)
        self.L, self.H, self.d = layers, heads, head_dim
        D = heads * head_dim
        self.D = D
        s = 1.0 / np.sqrt(D)
        self.Wk = rng.standard_normal((layers, D, D)) * s
        self.Wv = rng.standard_normal((layers, D, D)) * s
        self.Wq = rng.standard_normal((layers, D, D)) * s
        self.Wo = rng.standard_normal((layers, D, out_vocab)) * s
        self.freq = rng.uniform(0.01, 1.0, D)
        self.phase = rng.uniform(0, 2 * np.pi, D)

    def embed(self, t):
        return np.sin(np.asarray(t, np.float64)[..., None] * self.freq + self.phase)

    def pos(self, j, shift=0.0):
        return np.cos(np.asarray(j, np.float64)[..., None] * self.freq * 0.1 + shift)

    def kv(self, tokens, positions, dtype=np.float32):
        """K/V rows [n, L, 2, H, d] for tokens at absolute positions."""
        e = self.embed(tokens)                                    # [n, D]
        k = np.einsum("nd,lde->nle", e, self.Wk) + self.pos(positions)[:, None, :]
        v = np.einsum("nd,lde->nle", e, self.Wv) + self.pos(positions, 1.0)[:, None, :]
        out = np.stack([k, v], axis=2).reshape(len(e), self.L, 2, self.H, self.d)
        return out.astype(dtype)

    def next_distribution(self, cache_kv, pending_token, pending_pos):
        """fp64 next-step distribution of the pending token given valid K/V rows."""
        own = self.kv([pending_token], [pending_pos]).astype(np.float64)
        kv = np.concatenate([np.asarray(cache_kv, np.float64), own], axis=0)
        e = self.embed([pending_token])[0]
        logits = np.zeros(self.Wo.shape[-1])
        for l in range(self.L):
            q = (e @ self.Wq[l] + self.pos(pending_pos)).reshape(self.H, self.d)
            K, Vv = kv[:, l, 0], kv[:, l, 1]                     # [n, H, d]
            sc = np.einsum("hd,nhd->hn", q, K) / np.sqrt(self.d)
            a = np.exp(sc - sc.max(axis=1, keepdims=True))
            a /= a.sum(axis=1, keepdims=True)
            ctx = np.einsum("hn,nhd->hd", a, Vv).reshape(-1)
            logits += ctx @ self.Wo[l]
        p = np.exp(logits - logits.max())
        return p / p.sum()


class PagedPayload:
    """K/V payload of a paged cache: [num_blocks, BS, L, 2, H, d]."""

    def __init__(self, model: ToyAttention, num_blocks, block_size, dtype=np.float32):
        self.m = model
        self.BS = block_size
        self.data = np.zeros((num_blocks, block_size, model.L, 2, model.H, model.d), dtype)

    def write(self, table_row, tokens, positions):
        rows = self.m.kv(tokens, positions, self.data.dtype)
        for r, j in zip(rows, positions):
            self.data[table_row[j // self.BS], j % self.BS] = r

    def gather(self, table_row, n):
        return np.stack([self.data[table_row[j // self.BS], j % self.BS] for j in range(n)]) \
            if n else np.zeros((0,) + self.data.shape[2:], self.data.dtype)
