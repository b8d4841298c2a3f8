"""Move a workload (numpy arrays from ``workloads``) into device tensors.

Rows are laid out [B][rows][ld] with ld padded so each row is a whole number
of 16-byte vectors, as the C ABI requires.  Pure data movement.
"""

from __future__ import annotations

import numpy as np
import torch

from .workloads import padded_ld


def rows_to_device(arr: np.ndarray, dtype: str, device, ld=None, pin=False) -> torch.Tensor:
    """[B][rows][V] numpy (bf16 bits as uint16, or fp32) -> [B][rows][ld] tensor."""
    B, R, V = arr.shape
    eb = 2 if dtype == "bf16" else 4
    ld = ld or padded_ld(V, eb)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    host = torch.zeros((B, R, ld), dtype=tdt, pin_memory=pin)
    src = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16) \
        if dtype == "bf16" else torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    host[:, :, :V] = src
    return host if device is None else host.to(device)


def to_device(inp: dict, device="cuda", pin=False) -> dict:
    """All verify inputs of a workload as tensors on `device` (None: host)."""
    dev = device

    def t(a, dt):
        x = torch.from_numpy(np.ascontiguousarray(a).astype(dt, copy=False))
        if pin:
            x = x.pin_memory()
        return x if dev is None else x.to(dev)

    extra = {}
    if inp.get("eos") is not None:
        extra["eos"] = t(inp["eos"], np.int32)
    if inp.get("max_new") is not None:
        extra["max_new"] = t(inp["max_new"], np.int32)
    if inp.get("top_k") is not None:
        extra["top_k"] = t(inp["top_k"], np.int32)
    if inp.get("rep_penalty") is not None:
        extra["rep_penalty"] = t(inp["rep_penalty"], np.float32)
        extra["rep_tokens"] = t(inp["rep_tokens"], np.int32)
    return dict(
        **extra,
        target=rows_to_device(inp["target"], inp["target_dtype"], dev, pin=pin),
        draft=rows_to_device(inp["draft"], inp["draft_dtype"], dev, pin=pin)
        if inp["draft"].shape[1] > 0 else None,
        draft_tokens=t(inp["tokens"], np.int32),
        k=t(inp["k"], np.int32),
        temperature=t(inp["temperature"], np.float32),
        top_p=t(inp["top_p"], np.float32),
        request_id=t(inp["request_id"].view(np.int32), np.int32),
        seq_len=t(inp["seq_len"], np.int32),
        seed=int(inp["seed"]),
        V=int(inp["target"].shape[-1]),
        draft_kind=inp["draft_kind"],
    )


def tree_to_device(inp: dict, device="cuda", pin=False) -> dict:
    """Token-tree inputs (workloads.tree_batch) as tensors on `device`."""
    def t(a, dt):
        x = torch.from_numpy(np.ascontiguousarray(a).astype(dt, copy=False))
        if pin:
            x = x.pin_memory()
        return x if device is None else x.to(device)

    extra = {}
    for key in ("top_k", "eos", "max_new"):
        if inp.get(key) is not None:
            extra[key] = t(inp[key], np.int32)
    if inp.get("rep_penalty") is not None:
        extra["rep_penalty"] = t(inp["rep_penalty"], np.float32)
        extra["rep_tokens"] = t(inp["rep_tokens"], np.int32)
    return dict(
        **extra,
        target=rows_to_device(inp["target"], inp["target_dtype"], device, pin=pin),
        draft=rows_to_device(inp["draft"], inp["draft_dtype"], device, pin=pin),
        parent=t(inp["parent"], np.int32),
        tokens=t(inp["tokens"], np.int32),
        n_nodes=t(inp["n"], np.int32),
        temperature=t(inp["temperature"], np.float32),
        top_p=t(inp["top_p"], np.float32),
        request_id=t(inp["request_id"].view(np.int32), np.int32),
        seq_len=t(inp["seq_len"], np.int32),
        seed=int(inp["seed"]),
        V=int(inp["target"].shape[-1]),
        draft_kind=inp["draft_kind"],
    )
