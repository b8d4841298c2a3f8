"""ctypes binding of libspecverify.so (the C ABI in include/spec_verify.h).

Argument marshalling only: every function passes device pointers of torch
tensors and the current CUDA stream to the library and raises on a non-zero
status.  No step of the verification or of the cache bookkeeping runs here,
and there is no fallback: if the library is missing the import fails loudly.

Functions carry the C names: sv_create, sv_destroy, sv_workspace_size,
spec_verify, bfl_init, bfl_reserve, bfl_fork_prefix, bfl_release,
kv_commit_rollback, kv_commit_draft, bfl_reserve_cow, kv_commit_copy,
kv_rollback_contig, sv_get_error.  ``Verifier`` and
``BlockPool`` are thin owners of a handle / workspace and of the pool arrays.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspecverify.so")

SV_OK, SV_ERR_INVALID, SV_ERR_OOM, SV_ERR_CUDA = 0, -1, -2, -3
SV_ERR_TIMEOUT, SV_ERR_UNSUPPORTED, SV_ERR_STATE, SV_ERR_TOO_LARGE = -4, -5, -6, -7
STATUS_NAMES = {0: "SV_OK", -1: "SV_ERR_INVALID", -2: "SV_ERR_OOM", -3: "SV_ERR_CUDA",
                -4: "SV_ERR_TIMEOUT", -5: "SV_ERR_UNSUPPORTED", -6: "SV_ERR_STATE",
                -7: "SV_ERR_TOO_LARGE"}
SV_STATIC_MAX_ROWS = 16384  # rows B * (kmax + 1) one spec_verify_static call accepts
SV_BF16, SV_FP32 = 0, 1
SV_DRAFT_LOGITS, SV_DRAFT_PROBS = 0, 1
ST_Q_ZERO, ST_BAD_INPUT, ST_RESIDUAL_EMPTY, ST_TIMEOUT = 1, 2, 4, 8
ST_EOS, ST_CAPPED = 16, 32
FLAG_NO_SKIP = 1
FLAG_TEST_WITHHOLD = 2  # testing aid: see SV_FLAG_TEST_WITHHOLD
FLAG_CLUSTER_PATH = 4   # force the cluster-resident kernel (see SV_FLAG_CLUSTER_PATH)
FLAG_STREAM_PATH = 8    # ask for the streaming kernel (see SV_FLAG_STREAM_PATH)
ROW_NONE, ROW_ACCEPTED, ROW_REJECTED, ROW_SKIPPED, ROW_INVALID, ROW_BONUS, ROW_TERMINAL = range(7)

EXPORTS = ("sv_verify_args_size", "sv_create", "sv_destroy", "sv_workspace_size",
           "spec_verify", "bfl_init", "bfl_reserve", "bfl_fork_prefix", "bfl_release",
           "kv_commit_rollback", "kv_rollback_contig", "sv_get_error", "spec_verify_static",
           "kv_commit_draft", "bfl_reserve_cow", "kv_commit_copy", "sv_tree_args_size",
           "spec_verify_tree", "kv_commit_tree")
SV_TREE_MAX_NODES = 4096


class KvPayload(ctypes.Structure):
    _fields_ = [("data", c_void_p), ("layers", c_int32), ("heads", c_int32),
                ("head_dim", c_int32), ("elem_bytes", c_int32)]


def _payload(kv: torch.Tensor) -> KvPayload:
    """kv: [num_blocks, layers, 2, heads, block_size, head_dim], contiguous."""
    if kv.dim() != 6 or kv.shape[2] != 2 or not kv.is_contiguous():
        raise ValueError("kv must be a contiguous [num_blocks, layers, 2, heads, BS, head_dim] tensor")
    p = KvPayload()
    p.data, p.layers, p.heads, p.head_dim = _ptr(kv), kv.shape[1], kv.shape[3], kv.shape[5]
    p.elem_bytes = kv.element_size()
    return p


class SvVerifyArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("kmax", c_int32), ("V", c_int32), ("flags", c_uint32),
                ("target", c_void_p), ("target_ld", c_int64),
                ("target_dtype", c_int32), ("draft_dtype", c_int32),
                ("draft_kind", c_int32), ("reserved0", c_int32),
                ("draft", c_void_p), ("draft_ld", c_int64),
                ("draft_tokens", c_void_p), ("k", c_void_p), ("temperature", c_void_p),
                ("top_p", c_void_p), ("request_id", c_void_p), ("seq_len", c_void_p),
                ("seed", c_uint64),
                ("accepted", c_void_p), ("out_tokens", c_void_p), ("num_emitted", c_void_p),
                ("status", c_void_p), ("debug", c_void_p), ("probs_p", c_void_p),
                ("probs_q", c_void_p), ("eos_id", c_void_p), ("max_new", c_void_p),
                ("rep_penalty", c_void_p), ("rep_tokens", c_void_p), ("rep_ld", c_int64),
                ("top_k", c_void_p)]


class SvTreeArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("N", c_int32), ("V", c_int32), ("flags", c_uint32),
                ("target", c_void_p), ("target_ld", c_int64),
                ("target_dtype", c_int32), ("draft_dtype", c_int32),
                ("draft_kind", c_int32), ("reserved0", c_int32),
                ("draft", c_void_p), ("draft_ld", c_int64),
                ("parent", c_void_p), ("tokens", c_void_p), ("n_nodes", c_void_p),
                ("temperature", c_void_p), ("top_p", c_void_p), ("top_k", c_void_p),
                ("request_id", c_void_p), ("seq_len", c_void_p), ("seed", c_uint64),
                ("accepted", c_void_p), ("path", c_void_p), ("out_tokens", c_void_p),
                ("num_emitted", c_void_p), ("status", c_void_p),
                ("eos_id", c_void_p), ("max_new", c_void_p),
                ("rep_penalty", c_void_p), ("rep_tokens", c_void_p), ("rep_ld", c_int64)]


class BflState(ctypes.Structure):
    _fields_ = [("num_blocks", c_int32), ("block_size", c_int32), ("free_stack", c_void_p),
                ("free_top", c_void_p), ("refcount", c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libspecverify.so; raises if it was not built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with __graft_entry__.build() "
                          "(the verification path has no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name in EXPORTS:
        getattr(lib, name)
    lib.sv_verify_args_size.restype = c_size_t
    lib.sv_create.argtypes = [ctypes.c_int, POINTER(c_void_p)]
    lib.sv_destroy.argtypes = [c_void_p]
    lib.sv_workspace_size.argtypes = [POINTER(SvVerifyArgs), POINTER(c_size_t)]
    lib.spec_verify.argtypes = [c_void_p, POINTER(SvVerifyArgs), c_void_p, c_size_t, c_void_p]
    lib.spec_verify_static.argtypes = [POINTER(SvVerifyArgs), c_void_p]
    lib.bfl_init.argtypes = [c_void_p, POINTER(BflState), c_void_p]
    lib.bfl_reserve.argtypes = [c_void_p, POINTER(BflState), c_int32, c_void_p, c_void_p,
                                c_void_p, c_int32, c_void_p]
    lib.bfl_fork_prefix.argtypes = [c_void_p, POINTER(BflState), c_int32, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_int32, c_int32, c_void_p]
    lib.bfl_release.argtypes = [c_void_p, POINTER(BflState), c_int32, c_void_p, c_void_p,
                                c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    lib.bfl_reserve_cow.argtypes = [c_void_p, POINTER(BflState), c_int32, c_void_p, c_void_p,
                                    c_void_p, c_int32, POINTER(KvPayload), c_void_p, c_void_p]
    lib.kv_commit_copy.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                   c_int32, c_int32, c_int32, c_void_p, POINTER(KvPayload), c_void_p]
    lib.kv_commit_draft.argtypes = [c_void_p, POINTER(BflState), c_int32, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_int32, c_void_p, c_void_p]
    lib.kv_commit_rollback.argtypes = [c_void_p, POINTER(BflState), c_int32, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_int32, c_void_p, c_void_p]
    lib.kv_rollback_contig.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_void_p]
    lib.sv_get_error.argtypes = [c_void_p, c_void_p, POINTER(c_int32)]
    lib.sv_tree_args_size.restype = c_size_t
    lib.spec_verify_tree.argtypes = [c_void_p, POINTER(SvTreeArgs), c_void_p]
    lib.kv_commit_tree.argtypes = [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                   POINTER(KvPayload), c_void_p]
    for name in EXPORTS[1:]:
        if name != "sv_tree_args_size":
            getattr(lib, name).restype = c_int32
    if lib.sv_verify_args_size() != ctypes.sizeof(SvVerifyArgs):
        raise ImportError("sv_verify_args layout mismatch between binding and library")
    if lib.sv_tree_args_size() != ctypes.sizeof(SvTreeArgs):
        raise ImportError("sv_tree_args layout mismatch between binding and library")
    _lib = lib
    return lib


class SvError(RuntimeError):
    def __init__(self, fn, code, detail=None):
        msg = f"{fn} returned {STATUS_NAMES.get(code, code)}"
        super().__init__(msg if detail is None else f"{msg}: {detail}")
        self.code = code


def _check(fn, code):
    if code != SV_OK:
        raise SvError(fn, code)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_FP32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _row_ld(t):
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError("expected [B][rows][ld] with a contiguous last dimension")
    return t.stride(1)


# --------------------------------------------------------------------------- #
# C-named functions
# --------------------------------------------------------------------------- #
def sv_create(device: int = 0) -> c_void_p:
    h = c_void_p()
    _check("sv_create", load_library().sv_create(device, ctypes.byref(h)))
    return h


def sv_destroy(handle) -> None:
    _check("sv_destroy", load_library().sv_destroy(handle))


def make_args(*, target, draft, draft_tokens, temperature, accepted, out_tokens, num_emitted,
              status, V=None, k=None, top_p=None, seed=0, request_id=None, seq_len=None,
              draft_kind="logits", flags=0, debug=None, probs_p=None, probs_q=None,
              eos=None, max_new=None, rep_penalty=None, rep_tokens=None, top_k=None):
    B, rows, _ = target.shape
    kmax = rows - 1
    a = SvVerifyArgs()
    a.B, a.kmax, a.V, a.flags = B, kmax, int(V if V is not None else target.shape[-1]), flags
    a.target, a.target_ld, a.target_dtype = _ptr(target), _row_ld(target), _dtype_code(target)
    if draft is not None and kmax > 0:
        a.draft, a.draft_ld, a.draft_dtype = _ptr(draft), _row_ld(draft), _dtype_code(draft)
    else:
        a.draft, a.draft_ld, a.draft_dtype = None, a.target_ld, a.target_dtype
    a.draft_kind = SV_DRAFT_PROBS if draft_kind == "probs" else SV_DRAFT_LOGITS
    a.draft_tokens = _ptr(draft_tokens) if kmax > 0 else None
    a.k, a.temperature, a.top_p = _ptr(k), _ptr(temperature), _ptr(top_p)
    a.request_id, a.seq_len, a.seed = _ptr(request_id), _ptr(seq_len), int(seed) & (2 ** 64 - 1)
    a.accepted, a.out_tokens = _ptr(accepted), _ptr(out_tokens)
    a.num_emitted, a.status = _ptr(num_emitted), _ptr(status)
    a.debug, a.probs_p, a.probs_q = _ptr(debug), _ptr(probs_p), _ptr(probs_q)
    a.eos_id, a.max_new = _ptr(eos), _ptr(max_new)
    a.rep_penalty, a.top_k = _ptr(rep_penalty), _ptr(top_k)
    if rep_tokens is not None:
        if rep_tokens.dim() != 2 or rep_tokens.stride(1) != 1:
            raise ValueError("rep_tokens must be [B][H] with unit stride along H")
        a.rep_tokens, a.rep_ld = _ptr(rep_tokens), rep_tokens.stride(0)
    else:
        a.rep_tokens, a.rep_ld = None, 0
    return a


def sv_workspace_size(args: SvVerifyArgs) -> int:
    n = c_size_t()
    _check("sv_workspace_size", load_library().sv_workspace_size(ctypes.byref(args), ctypes.byref(n)))
    return n.value


def spec_verify(handle, args: SvVerifyArgs, workspace: torch.Tensor, stream=None) -> None:
    _check("spec_verify", load_library().spec_verify(handle, ctypes.byref(args), _ptr(workspace),
                                                     workspace.numel() * workspace.element_size(),
                                                     _stream(stream)))


def spec_verify_static(args: SvVerifyArgs, stream=None) -> None:
    """spec_verify without a handle or workspace, for callers that cannot
    allocate device memory (inside an allocator hook, or a runtime that owns
    all memory up front): its scratch is a fixed per-device array in the
    library, shared by every call and kept between calls, so calls must not
    overlap on the GPU.  At most SV_STATIC_MAX_ROWS rows B * (kmax + 1), else
    SvError(SV_ERR_TOO_LARGE).  The first call on a device does a one-time
    set-up; make it before any stream capture."""
    code = load_library().spec_verify_static(ctypes.byref(args), _stream(stream))
    if code == SV_ERR_TOO_LARGE:
        raise SvError("spec_verify_static", code,
                      f"B * (kmax + 1) = {args.B * (args.kmax + 1)} rows exceeds the fixed "
                      f"scratch of {SV_STATIC_MAX_ROWS} rows")
    _check("spec_verify_static", code)


def _state(pool) -> BflState:
    s = BflState()
    s.num_blocks, s.block_size = pool.num_blocks, pool.block_size
    s.free_stack, s.free_top, s.refcount = (_ptr(pool.free_stack), _ptr(pool.free_top),
                                            _ptr(pool.refcount))
    return s


def bfl_init(handle, pool, stream=None) -> None:
    _check("bfl_init", load_library().bfl_init(handle, ctypes.byref(_state(pool)), _stream(stream)))


def bfl_reserve(handle, pool, seq_len, k, block_table, stream=None) -> None:
    _check("bfl_reserve", load_library().bfl_reserve(
        handle, ctypes.byref(_state(pool)), seq_len.shape[0], _ptr(seq_len), _ptr(k),
        _ptr(block_table), block_table.shape[1], _stream(stream)))


def bfl_fork_prefix(handle, pool, src, dst, n_blocks, block_table, stream=None) -> None:
    _check("bfl_fork_prefix", load_library().bfl_fork_prefix(
        handle, ctypes.byref(_state(pool)), src.shape[0], _ptr(src), _ptr(dst), _ptr(n_blocks),
        _ptr(block_table), block_table.shape[0], block_table.shape[1], _stream(stream)))


def bfl_release(handle, pool, req_ids, seq_len, block_table, n_freed=None, stream=None) -> None:
    _check("bfl_release", load_library().bfl_release(
        handle, ctypes.byref(_state(pool)), req_ids.shape[0], _ptr(req_ids), _ptr(seq_len),
        _ptr(block_table), block_table.shape[0], block_table.shape[1], _ptr(n_freed),
        _stream(stream)))


def bfl_reserve_cow(handle, pool, seq_len, k, block_table, kv, cow_scratch, stream=None) -> None:
    """cow_scratch: int32 device tensor of at least 3 * B elements (caller-owned)."""
    if cow_scratch.numel() < 3 * seq_len.numel():
        raise ValueError("cow_scratch needs 3 * B int32 elements")
    _check("bfl_reserve_cow", load_library().bfl_reserve_cow(
        handle, ctypes.byref(_state(pool)), seq_len.numel(), _ptr(seq_len), _ptr(k),
        _ptr(block_table), block_table.shape[1], ctypes.byref(_payload(kv)), _ptr(cow_scratch),
        _stream(stream)))


def kv_commit_copy(handle, accepted, seq_len, block_table, block_size, num_blocks, stage, kv,
                   stream=None) -> None:
    """stage: [B, kmax + 1, layers, 2, heads, head_dim] contiguous, kv's dtype."""
    if stage.dim() != 6 or not stage.is_contiguous() or stage.dtype != kv.dtype:
        raise ValueError("stage must be a contiguous [B, kmax+1, layers, 2, heads, head_dim] tensor")
    _check("kv_commit_copy", load_library().kv_commit_copy(
        handle, accepted.numel(), stage.shape[1] - 1, _ptr(accepted), _ptr(seq_len),
        _ptr(block_table), block_table.shape[1], block_size, num_blocks, _ptr(stage),
        ctypes.byref(_payload(kv)), _stream(stream)))


def make_tree_args(*, target, draft, parent, tokens, temperature, accepted, path, out_tokens,
                   num_emitted, status, V=None, n_nodes=None, top_p=None, top_k=None, seed=0,
                   request_id=None, seq_len=None, draft_kind="logits", eos=None,
                   max_new=None, rep_penalty=None, rep_tokens=None) -> SvTreeArgs:
    """target, draft: [B, N+1, ld] rows per tree node; parent, tokens: [B, N] int32."""
    B, rows, _ = target.shape
    a = SvTreeArgs()
    a.B, a.N, a.V, a.flags = B, rows - 1, int(V if V is not None else target.shape[-1]), 0
    a.target, a.target_ld, a.target_dtype = _ptr(target), _row_ld(target), _dtype_code(target)
    a.draft, a.draft_ld, a.draft_dtype = _ptr(draft), _row_ld(draft), _dtype_code(draft)
    a.draft_kind = SV_DRAFT_PROBS if draft_kind == "probs" else SV_DRAFT_LOGITS
    a.parent, a.tokens, a.n_nodes = _ptr(parent), _ptr(tokens), _ptr(n_nodes)
    a.temperature, a.top_p, a.top_k = _ptr(temperature), _ptr(top_p), _ptr(top_k)
    a.request_id, a.seq_len, a.seed = _ptr(request_id), _ptr(seq_len), int(seed) & (2 ** 64 - 1)
    a.accepted, a.path, a.out_tokens = _ptr(accepted), _ptr(path), _ptr(out_tokens)
    a.num_emitted, a.status = _ptr(num_emitted), _ptr(status)
    a.eos_id, a.max_new = _ptr(eos), _ptr(max_new)
    a.rep_penalty = _ptr(rep_penalty)
    if rep_tokens is not None:
        if rep_tokens.dim() != 2 or rep_tokens.stride(1) != 1:
            raise ValueError("rep_tokens must be [B][H] with unit stride along H")
        a.rep_tokens, a.rep_ld = _ptr(rep_tokens), rep_tokens.stride(0)
    else:
        a.rep_tokens, a.rep_ld = None, 0
    return a


def spec_verify_tree(handle, args: SvTreeArgs, stream=None) -> None:
    _check("spec_verify_tree", load_library().spec_verify_tree(handle, ctypes.byref(args),
                                                               _stream(stream)))


def kv_commit_tree(handle, accepted, path, seq_len, block_table, block_size, num_blocks, stage,
                   kv, max_depth, stream=None) -> None:
    """stage: [B, N + 1, layers, 2, heads, head_dim] contiguous (one entry per
    tree node); path: [B, N] from spec_verify_tree."""
    if stage.dim() != 6 or not stage.is_contiguous() or stage.dtype != kv.dtype:
        raise ValueError("stage must be a contiguous [B, N+1, layers, 2, heads, head_dim] tensor")
    _check("kv_commit_tree", load_library().kv_commit_tree(
        handle, accepted.numel(), stage.shape[1] - 1, int(max_depth), _ptr(accepted), _ptr(path),
        _ptr(seq_len), _ptr(block_table), block_table.shape[1], block_size, num_blocks,
        _ptr(stage), ctypes.byref(_payload(kv)), _stream(stream)))


def kv_commit_draft(handle, pool, seq_len, accepted, draft_len, draft_table, n_freed=None,
                    stream=None) -> None:
    _check("kv_commit_draft", load_library().kv_commit_draft(
        handle, ctypes.byref(_state(pool)), draft_len.numel(), _ptr(seq_len), _ptr(accepted),
        _ptr(draft_len), _ptr(draft_table), draft_table.shape[1], _ptr(n_freed), _stream(stream)))


def kv_commit_rollback(handle, pool, k, accepted, seq_len, block_table, n_freed=None,
                       stream=None) -> None:
    _check("kv_commit_rollback", load_library().kv_commit_rollback(
        handle, ctypes.byref(_state(pool)), accepted.shape[0], _ptr(k), _ptr(accepted),
        _ptr(seq_len), _ptr(block_table), block_table.shape[1], _ptr(n_freed), _stream(stream)))


def kv_rollback_contig(handle, accepted, write_ptr, stream=None) -> None:
    _check("kv_rollback_contig", load_library().kv_rollback_contig(
        handle, accepted.shape[0], _ptr(accepted), _ptr(write_ptr), _stream(stream)))


def sv_get_error(handle, stream=None) -> int:
    code = c_int32()
    _check("sv_get_error", load_library().sv_get_error(handle, _stream(stream), ctypes.byref(code)))
    return code.value


# --------------------------------------------------------------------------- #
# owners
# --------------------------------------------------------------------------- #
class BlockPool:
    """Device arrays of a block pool (free stack, top, refcounts) + bfl_init."""

    def __init__(self, handle, num_blocks: int, block_size: int, device="cuda", stream=None):
        self.handle = handle
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.free_stack = torch.empty(max(1, num_blocks), dtype=torch.int32, device=device)
        self.free_top = torch.empty(1, dtype=torch.int32, device=device)
        self.refcount = torch.empty(max(1, num_blocks), dtype=torch.int32, device=device)
        bfl_init(handle, self, stream)

    def reserve(self, seq_len, k, block_table, stream=None):
        bfl_reserve(self.handle, self, seq_len, k, block_table, stream)

    def commit_rollback(self, k, accepted, seq_len, block_table, n_freed=None, stream=None):
        kv_commit_rollback(self.handle, self, k, accepted, seq_len, block_table, n_freed, stream)

    def reserve_cow(self, seq_len, k, block_table, kv, cow_scratch, stream=None):
        bfl_reserve_cow(self.handle, self, seq_len, k, block_table, kv, cow_scratch, stream)

    def commit_draft(self, seq_len, accepted, draft_len, draft_table, n_freed=None, stream=None):
        kv_commit_draft(self.handle, self, seq_len, accepted, draft_len, draft_table, n_freed, stream)

    def fork_prefix(self, src, dst, n_blocks, block_table, stream=None):
        bfl_fork_prefix(self.handle, self, src, dst, n_blocks, block_table, stream)

    def release(self, req_ids, seq_len, block_table, n_freed=None, stream=None):
        bfl_release(self.handle, self, req_ids, seq_len, block_table, n_freed, stream)


class Verifier:
    """A handle plus a lazily grown, zero-initialised workspace."""

    def __init__(self, device: int = 0):
        self.device = torch.device("cuda", device)
        self.handle = sv_create(device)
        self.workspace = None
        self.path_flags = 0  # kernel selection added to every verify() call

    def close(self):
        if self.handle is not None:
            sv_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def ensure_workspace(self, args: SvVerifyArgs):
        need = sv_workspace_size(args)
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self.workspace

    def outputs(self, B: int, kmax: int):
        d = self.device
        return dict(accepted=torch.empty(B, dtype=torch.int32, device=d),
                    out_tokens=torch.empty(B, kmax + 1, dtype=torch.int32, device=d),
                    num_emitted=torch.empty(B, dtype=torch.int32, device=d),
                    status=torch.empty(B, dtype=torch.int32, device=d))

    def verify(self, *, target, draft, draft_tokens, temperature, out=None, stream=None, **kw):
        """Run spec_verify; returns the output tensors (allocated unless given).
        The handle's `path_flags` (kernel selection, 0 by default) are added
        to the call's flags."""
        B, rows, _ = target.shape
        out = out or self.outputs(B, rows - 1)
        kw["flags"] = int(kw.get("flags", 0)) | self.path_flags
        a = make_args(target=target, draft=draft, draft_tokens=draft_tokens,
                      temperature=temperature, **out, **kw)
        ws = self.ensure_workspace(a)
        spec_verify(self.handle, a, ws, stream)
        return out

    def tree_outputs(self, B: int, N: int):
        d = self.device
        return dict(accepted=torch.empty(B, dtype=torch.int32, device=d),
                    path=torch.empty(B, max(N, 1), dtype=torch.int32, device=d),
                    out_tokens=torch.empty(B, N + 1, dtype=torch.int32, device=d),
                    num_emitted=torch.empty(B, dtype=torch.int32, device=d),
                    status=torch.empty(B, dtype=torch.int32, device=d))

    def verify_tree(self, *, target, draft, parent, tokens, temperature, out=None, stream=None,
                    **kw):
        """Run spec_verify_tree; returns the output tensors (allocated unless given)."""
        B, rows, _ = target.shape
        out = out or self.tree_outputs(B, rows - 1)
        a = make_tree_args(target=target, draft=draft, parent=parent, tokens=tokens,
                           temperature=temperature, **out, **kw)
        spec_verify_tree(self.handle, a, stream)
        return out

    def error(self, stream=None) -> int:
        return sv_get_error(self.handle, stream)
