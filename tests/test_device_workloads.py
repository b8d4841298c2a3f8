"""Host checks of the throughput-input module: the byte counts behind every
GB/s and roofline fraction the bench reports, and the simulated draft
sampler's law (top-p cut, greedy ties), run with torch on the CPU."""

import math

import numpy as np
import torch

from speculative_decoding_verification_07_gb300 import device_workloads as DW


def _batch(k, V, draft_kind="logits"):
    """A CPU batch with ragged k (a list)."""
    return DW.make_batch(len(k), torch.tensor(k), V, device="cpu", seed=11, temperature=0.8,
                         top_p=0.9, draft_kind=draft_kind)


def test_full_bytes_counts_every_row_and_the_metadata():
    # ragged k = (1, 3, 0): target rows k+1, draft rows k, 2-byte target, 4-byte probs
    k, V = [1, 3, 0], 40
    b = _batch(k, V, draft_kind="probs")
    rows = sum((kb + 1) * V * 2 + kb * V * 4 for kb in k)
    meta = sum(4 * kb + 4 * (kb + 1) + 24 for kb in k)
    assert DW.full_bytes(b) == rows + meta


def test_full_bytes_at_the_metric_shape():
    # B=64, k=4, V=128256, bf16 target and draft: 82.08 MB + 65.67 MB of rows
    V = 128256
    b = {"target": torch.empty(1, 1, V, dtype=torch.bfloat16),
         "draft": torch.empty(1, 1, V, dtype=torch.bfloat16),
         "k": torch.full((64,), 4, dtype=torch.int32)}
    rows = 64 * (5 * V * 2 + 4 * V * 2)
    assert DW.full_bytes(b) == rows + 64 * (16 + 20 + 24)
    assert abs(64 * 5 * V * 2 / 1e6 - 82.08) < 0.01 and abs(64 * 4 * V * 2 / 1e6 - 65.67) < 0.01


def test_needed_bytes_stop_at_the_first_rejection():
    k, V = [2, 3, 3, 0], 16
    b = _batch(k, V)
    # a = -1 (invalid: row 0 still read), 0 (rejected at row 0), 3 = k (all accepted: bonus row,
    # no draft row past k), 0 with k = 0 (bonus only)
    acc = torch.tensor([-1, 0, 3, 0])
    want = (1 * V * 2 + 1 * V * 2) + (1 * V * 2 + 1 * V * 2) + (4 * V * 2 + 3 * V * 2) + (1 * V * 2)
    assert DW.needed_bytes(b, acc) == want
    assert DW.needed_bytes(b, acc) <= DW.full_bytes(b)


def test_sets_for_exceeds_the_floor_within_the_cap():
    floor = 400 << 20
    for per in (1, 45 << 10, 4_610_000, 147_750_000, 700_100_000, 9 << 30):
        n = DW.sets_for(per)
        assert 1 <= n <= 16
        if n < 16:
            assert n * per >= floor and (n == 1 or (n - 1) * per < floor)
    assert DW.sets_for(147_750_000) == 3


def test_make_batch_shapes_and_ranges():
    b = DW.make_batch(5, torch.tensor([0, 1, 4, 2, 4]), 300, device="cpu", seed=3, top_p=0.95,
                      draft_kind="probs")
    assert b["target"].shape == (5, 5, 300) and b["target"].dtype == torch.bfloat16
    assert b["draft"].shape == (5, 4, 300) and b["draft"].dtype == torch.float32
    assert torch.allclose(b["draft"].sum(-1), torch.ones(5, 4), atol=1e-5)
    t = b["draft_tokens"]
    assert t.dtype == torch.int32 and int(t.min()) >= 0 and int(t.max()) < 300
    assert 128 <= int(b["seq_len"].min()) and int(b["seq_len"].max()) <= 8192
    # the same seed gives the same batch
    b2 = DW.make_batch(5, torch.tensor([0, 1, 4, 2, 4]), 300, device="cpu", seed=3, top_p=0.95,
                       draft_kind="probs")
    assert torch.equal(b["target"], b2["target"]) and torch.equal(t, b2["draft_tokens"])


def test_sampler_top_p_keeps_the_smallest_prefix_reaching_p():
    # softmax of these logits: 0.5, 0.25, 0.125, 0.125 (T = 1); top-p 0.7 keeps the first two
    x = torch.log(torch.tensor([[0.5, 0.25, 0.125, 0.125]]))
    rows = x.repeat(4000, 1)
    g = torch.Generator().manual_seed(5)
    tok = DW._sample_rows(rows, torch.ones(4000), torch.full((4000,), 0.7), g)
    counts = np.bincount(tok.numpy(), minlength=4)
    assert counts[2] == 0 and counts[3] == 0
    # within the kept set the law is renormalised: 2/3 and 1/3 (4000 draws: sd ~ 0.0075)
    assert abs(counts[0] / 4000 - 2 / 3) < 0.04
    # top-p = 1 keeps everything
    tok = DW._sample_rows(rows, torch.ones(4000), torch.ones(4000), g)
    assert np.bincount(tok.numpy(), minlength=4)[3] > 0


def test_sampler_greedy_picks_only_among_tied_maxima():
    x = torch.tensor([[1.0, 3.0, -2.0, 3.0, 0.5]]).repeat(2000, 1)
    g = torch.Generator().manual_seed(9)
    tok = DW._sample_rows(x, torch.zeros(2000), torch.ones(2000), g)
    counts = np.bincount(tok.numpy(), minlength=5)
    assert counts[0] == counts[2] == counts[4] == 0
    assert min(counts[1], counts[3]) > 800  # both tied maxima are drawn


def test_sampler_probability_rows_match_their_logits():
    # a row of probabilities is sampled through its logarithm: same law as the logits
    p = torch.tensor([[0.1, 0.6, 0.3]])
    g1, g2 = torch.Generator().manual_seed(1), torch.Generator().manual_seed(1)
    a = DW._sample_rows(p.repeat(500, 1), torch.ones(500), torch.ones(500), g1, probs=True)
    b = DW._sample_rows(torch.log(p).repeat(500, 1), torch.ones(500), torch.ones(500), g2)
    assert torch.equal(a, b)
    assert math.isclose(float((a == 1).float().mean()), 0.6, abs_tol=0.07)
