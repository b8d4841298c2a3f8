"""Seeded synthetic inputs built directly on the GPU, for throughput runs.

The parity tests use the numpy generators in workloads.py (the oracle reads
them on the host).  Throughput runs at the largest configurations (up to
B=1024 x 9 rows x V=256000) would take minutes to synthesise on the host, so
this module builds the same recipes with torch on the device: i.i.d. normal
target logits, draft logits (or fp32 probabilities) = target + normal noise,
per-request temperature / top-p / ragged k, and proposals drawn from the
draft's own transformed distribution (the simulated draft model's sampler:
softmax(z / T), top-p, one multinomial draw per row; T = 0 picks uniformly
among tied maxima).  It holds none of the verifier's arithmetic.
"""

from __future__ import annotations

import math

import torch


def _sample_rows(logits: torch.Tensor, T: torch.Tensor, top_p: torch.Tensor, gen,
                 probs: bool = False, chunk: int = 512) -> torch.Tensor:
    """One draw per row of a [R, V] fp32 tensor from top-p(softmax(row / T))
    (rows of probabilities are taken in log space first)."""
    R, V = logits.shape
    out = torch.empty(R, dtype=torch.int64, device=logits.device)
    for r0 in range(0, R, chunk):
        x = logits[r0:r0 + chunk].float()
        if probs:
            x = torch.log(x)
        t = T[r0:r0 + chunk].float().unsqueeze(1)
        p = top_p[r0:r0 + chunk].float().unsqueeze(1)
        greedy = (t == 0).squeeze(1)
        z = torch.where(t > 0, x / torch.where(t > 0, t, torch.ones_like(t)), x)
        w = torch.softmax(z, dim=1)
        sw, idx = torch.sort(w, dim=1, descending=True)
        c = torch.cumsum(sw, dim=1)
        keep = (c - sw) < p                       # tokens up to the one that reaches top_p
        sw = torch.where(keep, sw, torch.zeros_like(sw))
        pick = torch.multinomial(sw, 1, generator=gen).squeeze(1)
        tok = idx.gather(1, pick.unsqueeze(1)).squeeze(1)
        if greedy.any():
            mx = x.max(dim=1, keepdim=True).values
            ties = (x == mx).float()
            g = torch.multinomial(ties, 1, generator=gen).squeeze(1)
            tok = torch.where(greedy, g, tok)
        out[r0:r0 + chunk] = tok
    return out


def make_batch(B: int, k, V: int, *, device, seed: int, target_sd: float = 3.0,
               draft_sd: float = 1.0, temperature=0.8, top_p=1.0, draft_kind: str = "logits",
               target_dtype=torch.bfloat16, draft_dtype=torch.bfloat16, kmax=None):
    """A batch as the C ABI takes it (torch tensors on `device`).

    k: an int (every request) or a [B] tensor (ragged).  temperature / top_p:
    a float or a [B] tensor.  draft_kind "probs": fp32 softmax(target +
    noise)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if isinstance(k, int):
        kk = torch.full((B,), k, dtype=torch.int32, device=device)
    else:
        kk = k.to(device=device, dtype=torch.int32)
    kmax = int(kk.max().item()) if kmax is None else kmax
    T = temperature if torch.is_tensor(temperature) else torch.full((B,), float(temperature))
    P = top_p if torch.is_tensor(top_p) else torch.full((B,), float(top_p))
    T, P = T.to(device=device, dtype=torch.float32), P.to(device=device, dtype=torch.float32)
    target = torch.empty(B, kmax + 1, V, dtype=target_dtype, device=device)
    draft = torch.empty(B, max(kmax, 1), V,
                        dtype=torch.float32 if draft_kind == "probs" else draft_dtype, device=device)
    tokens = torch.zeros(B, max(kmax, 1), dtype=torch.int32, device=device)
    for b0 in range(0, B, 64):
        b1 = min(B, b0 + 64)
        t = torch.randn(b1 - b0, kmax + 1, V, generator=gen, device=device) * target_sd
        target[b0:b1] = t.to(target_dtype)
        tq = target[b0:b1, :max(kmax, 1)].float()
        d = tq + torch.randn(tq.shape, generator=gen, device=device) * draft_sd
        if draft_kind == "probs":
            d = torch.softmax(d, dim=2)
            draft[b0:b1] = d
        else:
            draft[b0:b1] = d.to(draft_dtype)
        if kmax > 0:
            rows = draft[b0:b1].reshape(-1, V)
            rT = T[b0:b1].repeat_interleave(max(kmax, 1))
            rP = P[b0:b1].repeat_interleave(max(kmax, 1))
            tok = _sample_rows(rows.float(), rT, rP, gen, probs=draft_kind == "probs")
            tokens[b0:b1] = tok.view(b1 - b0, max(kmax, 1)).to(torch.int32)
    seq = torch.randint(128, 8193, (B,), generator=gen, device=device, dtype=torch.int32)
    return dict(target=target, draft=draft, draft_tokens=tokens, k=kk, temperature=T, top_p=P,
                seq_len=seq, request_id=torch.arange(B, dtype=torch.int32, device=device),
                seed=seed + 7, draft_kind=draft_kind, kmax=kmax)


def full_bytes(batch) -> int:
    """Every target row (k_b + 1) and draft row (k_b) of the batch, plus the
    per-request metadata read and written."""
    V = batch["target"].shape[-1]
    st, sd = batch["target"].element_size(), batch["draft"].element_size()
    k = batch["k"].long()
    rows = ((k + 1) * V * st + k * V * sd).sum().item()
    return int(rows + (4 * k + 4 * (k + 1) + 24).sum().item())


def needed_bytes(batch, accepted) -> int:
    """The rows the method must read: target rows 0..a_b and draft rows
    0..min(a_b, k_b - 1)."""
    V = batch["target"].shape[-1]
    st, sd = batch["target"].element_size(), batch["draft"].element_size()
    k = batch["k"].long()
    a = accepted.long().clamp(min=0)
    return int(((a + 1) * V * st + torch.minimum(a + 1, k) * V * sd).sum().item())


def sets_for(nbytes_per_set: int, floor_bytes: int = 400 << 20, cap: int = 16) -> int:
    """How many input sets to rotate so that a run touches more than
    `floor_bytes` (several times the L2) between reuses."""
    return max(1, min(cap, math.ceil(floor_bytes / max(1, nbytes_per_set))))
