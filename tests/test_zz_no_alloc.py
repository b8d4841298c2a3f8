"""spec_verify_static (the entry point for callers that cannot allocate device
memory) against spec_verify, through the C ABI.

Two different batches go through spec_verify_static back to back on one
stream, so the second call runs on the scratch array the first one left
behind; both must give what spec_verify gives for the same arguments.  The
file is named to be collected last, and it builds the library itself, so it
passes both alone in a fresh process and after the other GPU tests.
"""

import os

import numpy as np
import pytest
import torch

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


def _outputs(ver, inp, probs):
    B, kmax, V = inp["tokens"].shape[0], inp["tokens"].shape[1], inp["target"].shape[-1]
    out = ver.outputs(B, kmax)
    for t in out.values():
        t.fill_(-7)
    if probs:
        out["probs_p"] = torch.full((B, kmax + 1, V), -1.0, device=ver.device)
        out["probs_q"] = torch.full((B, max(kmax, 1), V), -1.0, device=ver.device)
    return out


def _same(ref, got, name):
    for key in ("accepted", "out_tokens", "num_emitted", "status"):
        assert torch.equal(ref[key], got[key]), f"{name}: {key} differs"
    for key in ("probs_p", "probs_q"):
        if key in ref:
            diff = (ref[key] - got[key]).abs().max().item()
            assert diff <= parity.PROB_TOL, f"{name}: {key} differs by {diff}"


def test_static_scratch_matches_workspace_path(ver):
    # (name, inputs, flags, per-row probabilities requested); the per-row
    # probabilities are compared only with row skipping off, since which rows
    # are skipped depends on timing
    opts = W.verify_b64_k4(B=32, V=32000)
    rng = np.random.default_rng(3)
    opts["top_k"] = rng.choice(np.array([0, 5, 50, 500], np.int32), 32)
    opts["eos"] = opts["tokens"][:, 1].copy()
    opts["max_new"] = rng.integers(1, 6, 32).astype(np.int32)
    opts["rep_penalty"] = rng.choice(np.array([1.0, 1.3], np.float32), 32)
    opts["rep_tokens"] = rng.integers(-1, 32000, (32, 40)).astype(np.int32)
    batches = [("verify B=64 k=4 V=128256 bf16", W.verify_b64_k4(), 0, False),
               ("paged bf16 V=32000, no skip", W.paged_bf16(), binding.FLAG_NO_SKIP, True),
               ("top-k, EOS, caps, repetition penalty", opts, 0, False)]
    devs = [device_io.to_device(inp, "cuda:0") for _, inp, _, _ in batches]

    # the existing entry point, with its own zero-filled workspace
    refs = []
    for dev, (_, inp, flags, probs) in zip(devs, batches):
        out = _outputs(ver, inp, probs)
        a = binding.make_args(**dev, **out, flags=flags)
        binding.spec_verify(ver.handle, a, ver.ensure_workspace(a))
        refs.append(out)
    torch.cuda.synchronize()
    assert ver.error() == 0

    # two calls in a row on one stream, sharing the fixed scratch array
    gots = []
    for dev, (_, inp, flags, probs) in zip(devs, batches):
        out = _outputs(ver, inp, probs)
        binding.spec_verify_static(binding.make_args(**dev, **out, flags=flags))
        gots.append(out)
    torch.cuda.synchronize()

    for ref, got, (name, _, _, _) in zip(refs, gots, batches):
        assert (ref["accepted"] >= 0).all(), name
        _same(ref, got, name)


def test_static_scratch_rejects_oversized_batch(ver):
    rows = binding.SV_STATIC_MAX_ROWS
    B, kmax, V = rows // 4 + 1, 3, 64  # B * (kmax + 1) = rows + 4
    d = ver.device
    target = torch.zeros(B, kmax + 1, V, dtype=torch.bfloat16, device=d)
    draft = torch.zeros(B, kmax, V, dtype=torch.bfloat16, device=d)
    out = ver.outputs(B, kmax)
    a = binding.make_args(target=target, draft=draft,
                          draft_tokens=torch.zeros(B, kmax, dtype=torch.int32, device=d),
                          temperature=torch.ones(B, device=d), **out)
    with pytest.raises(binding.SvError) as e:
        binding.spec_verify_static(a)
    assert e.value.code == binding.SV_ERR_TOO_LARGE
    assert "exceeds" in str(e.value)
