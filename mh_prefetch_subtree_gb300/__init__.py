"""Python binding of libps (scoring and walking one prefetched subtree batch).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libps.so``; this module turns torch tensors into the C structs
of ``include/ps.h`` and calls the entry points of the same names.  There is
no CPU fallback: if the library is missing or fails to load, every call
raises.

Entry points (see include/ps.h for the contract):
    ps_score_workspace_bytes, ps_score_subtree, ps_score_rows,
    ps_assemble_subtree, ps_walk_subtree, ps_score_walk_subtree, ps_carry_state,
    ps_validate_subtree,
    ps_score_subtree_noalloc, ps_status_string, ps_version
Convenience: ``make_batch``, ``make_score_out``, ``make_tree``,
``make_walk_out`` build the structs from tensors; ``DeviceSubtree`` holds a
whole batch on the GPU with its outputs and workspace.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libps.so")

PS_OK = 0
PS_FLAG_MASKED_LOGITS = 0x1
PS_ERR_INVALID_ARG, PS_ERR_INFEASIBLE, PS_ERR_BAD_TREE, PS_ERR_UNSUPPORTED = 1, 2, 3, 4
PS_ERR_CUDA, PS_ERR_TIMEOUT, PS_ERR_WORKSPACE = 5, 6, 7
PS_BF16, PS_F32 = 0, 1
PS_DEV_BITS = {
    0x01: "BAD_TOKEN", 0x02: "NONFINITE", 0x04: "INFEASIBLE", 0x08: "BAD_TREE",
    0x10: "BAD_LAYOUT", 0x20: "TIMEOUT", 0x40: "BAD_ROW_INDEX", 0x80: "BAD_UNIFORM",
}
PS_NODE_LEAF, PS_NODE_DEFERRED = -1, -2

_vp = ctypes.c_void_p


class PsSubtreeBatch(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int32), ("T", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("n_chains", ctypes.c_int32), ("n_seg", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("n_rows", ctypes.c_int64),
                ("ld", ctypes.c_int64), ("n_logit_rows", ctypes.c_int64),
                ("alpha", ctypes.c_double), ("tau", ctypes.c_double),
                ("eps", ctypes.c_double), ("chain_seg0", _vp), ("seg_row0", _vp), ("seg_cut", _vp), ("seg_src", _vp),
                ("logits", _vp), ("row_index", _vp), ("tokens", _vp),
                ("root_lp0", _vp), ("root_lq", _vp)]


class PsScoreOut(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("lp0", "lq", "lp_y", "lq_y", "lp_x", "lq_x",
                                   "log_ratio", "log_accept", "status", "entropy",
                                   "eps_class")]


class PsTree(ctypes.Structure):
    _fields_ = [("n_chains", ctypes.c_int32), ("n_nodes", ctypes.c_int32),
                ("n_seg", ctypes.c_int32), ("max_steps", ctypes.c_int32),
                ("chain_node0", _vp), ("chain_seg0", _vp), ("acc", _vp), ("rej", _vp),
                ("req", _vp), ("u", _vp)]


class PsWalkOut(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("state_seg", "end_node", "k_delta", "path", "status")]


class PsCarryIo(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("state_seg", "row_lp0", "row_lq", "row_entropy", "prev_lp0",
                                   "prev_lq", "prev_entropy", "next_lp0", "next_lq",
                                   "next_entropy", "loglik", "confidence", "status")]


class PsError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {ps_status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libps.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libps.so is not built ({LIB_PATH}); run "
                               "`python -m mh_prefetch_subtree_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.ps_score_workspace_bytes.argtypes = [ctypes.POINTER(PsSubtreeBatch)]
        L.ps_score_workspace_bytes.restype = ctypes.c_size_t
        L.ps_score_subtree.argtypes = [ctypes.POINTER(PsSubtreeBatch), ctypes.POINTER(PsScoreOut),
                                       _vp, ctypes.c_size_t, _vp]
        L.ps_score_subtree.restype = ctypes.c_int
        L.ps_score_rows.argtypes = [ctypes.POINTER(PsSubtreeBatch), _vp, _vp, _vp, _vp, _vp,
                                    ctypes.c_size_t, _vp]
        L.ps_score_rows.restype = ctypes.c_int
        L.ps_score_rows_multi.argtypes = [ctypes.POINTER(PsSubtreeBatch),
                                          ctypes.POINTER(ctypes.c_double), ctypes.c_int32,
                                          _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.ps_score_rows_multi.restype = ctypes.c_int
        L.ps_assemble_subtree.argtypes = [ctypes.POINTER(PsSubtreeBatch), _vp, _vp,
                                          ctypes.POINTER(PsScoreOut), _vp]
        L.ps_assemble_subtree.restype = ctypes.c_int
        L.ps_score_subtree_noalloc.argtypes = [ctypes.POINTER(PsSubtreeBatch),
                                               ctypes.POINTER(PsScoreOut), _vp]
        L.ps_score_subtree_noalloc.restype = ctypes.c_int
        L.ps_walk_subtree.argtypes = [ctypes.POINTER(PsTree), _vp, ctypes.POINTER(PsWalkOut), _vp]
        L.ps_walk_subtree.restype = ctypes.c_int
        L.ps_score_walk_subtree.argtypes = [ctypes.POINTER(PsSubtreeBatch), ctypes.POINTER(PsTree),
                                            ctypes.POINTER(PsScoreOut), ctypes.POINTER(PsWalkOut),
                                            _vp, ctypes.c_size_t, _vp]
        L.ps_score_walk_subtree.restype = ctypes.c_int
        L.ps_carry_state.argtypes = [ctypes.POINTER(PsSubtreeBatch), ctypes.POINTER(PsCarryIo),
                                     _vp]
        L.ps_carry_state.restype = ctypes.c_int
        i32p = ctypes.POINTER(ctypes.c_int32)
        L.ps_build_bfs_tree.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32] + \
            [_vp] * 7 + [i32p, i32p, i32p]
        L.ps_build_bfs_tree.restype = ctypes.c_int
        L.ps_predictive_allocation.argtypes = [ctypes.c_int32, _vp, _vp, _vp, _vp,
                                               ctypes.c_int32, ctypes.POINTER(ctypes.c_double),
                                               _vp]
        L.ps_predictive_allocation.restype = ctypes.c_int
        L.ps_midpoint_branch_probability.argtypes = [ctypes.c_double, ctypes.c_double]
        L.ps_midpoint_branch_probability.restype = ctypes.c_double
        L.ps_validate_subtree.argtypes = [ctypes.POINTER(PsSubtreeBatch), ctypes.POINTER(PsTree),
                                          ctypes.c_char_p, ctypes.c_size_t]
        L.ps_validate_subtree.restype = ctypes.c_int
        L.ps_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp, _vp]
        L.ps_selftest_wait_timeout.restype = ctypes.c_int
        L.ps_selftest_read.argtypes = [_vp, ctypes.c_size_t, _vp, _vp]
        L.ps_selftest_read.restype = ctypes.c_int
        L.ps_status_string.argtypes = [ctypes.c_int]
        L.ps_status_string.restype = ctypes.c_char_p
        L.ps_version.argtypes = []
        L.ps_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def ps_status_string(status: int) -> str:
    return lib().ps_status_string(int(status)).decode()


def ps_version() -> str:
    return lib().ps_version().decode()


def ps_score_workspace_bytes(batch: PsSubtreeBatch) -> int:
    return int(lib().ps_score_workspace_bytes(ctypes.byref(batch)))


def ps_score_subtree(batch: PsSubtreeBatch, out: PsScoreOut, workspace: torch.Tensor,
                     stream=None, check: bool = True) -> int:
    ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = lib().ps_score_subtree(ctypes.byref(batch), ctypes.byref(out), ws_ptr, ws_bytes,
                                _stream(stream, workspace))
    if check and st != PS_OK:
        raise PsError(st, "ps_score_subtree")
    return st


def ps_score_subtree_noalloc(batch: PsSubtreeBatch, out: PsScoreOut, stream=None,
                             check: bool = True) -> int:
    """Scoring for callers that cannot allocate device memory: no workspace
    argument; libps uses its own static device array (see include/ps.h for the
    row limit, the once-per-device set-up and why overlapping calls race)."""
    st = lib().ps_score_subtree_noalloc(ctypes.byref(batch), ctypes.byref(out),
                                        _stream(stream, None))
    if check and st != PS_OK:
        raise PsError(st, "ps_score_subtree_noalloc")
    return st


def ps_score_rows(batch: PsSubtreeBatch, lp0: torch.Tensor, lq: torch.Tensor,
                  status: torch.Tensor, workspace: torch.Tensor, stream=None,
                  check: bool = True, entropy: torch.Tensor | None = None) -> int:
    _need(lp0, torch.float64, "lp0")
    _need(lq, torch.float64, "lq")
    _need(entropy, torch.float64, "entropy", optional=True)
    _need(status, torch.int32, "status")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().ps_score_rows(ctypes.byref(batch), _ptr(lp0), _ptr(lq), _ptr(entropy),
                             _ptr(status), _ptr(workspace), ws_bytes, _stream(stream, workspace))
    if check and st != PS_OK:
        raise PsError(st, "ps_score_rows")
    return st


def ps_score_rows_multi(batch: PsSubtreeBatch, taus, lp0: torch.Tensor, lq: torch.Tensor,
                        status: torch.Tensor, workspace: torch.Tensor, stream=None,
                        check: bool = True, entropy: torch.Tensor | None = None) -> int:
    """log p0 and log q_tau for several temperatures in one pass (each 1/tau
    in {1, 2, 4, 8}); lq is [len(taus), n_rows]."""
    taus = [float(t) for t in taus]
    _need(lp0, torch.float64, "lp0")
    _need(lq, torch.float64, "lq")
    _need(entropy, torch.float64, "entropy", optional=True)
    _need(status, torch.int32, "status")
    if len(lq.shape) != 2 or lq.shape[0] != len(taus) or lq.shape[1] != lp0.shape[0]:
        raise ValueError("lq must be [len(taus), n_rows]")
    arr = (ctypes.c_double * max(1, len(taus)))(*taus)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().ps_score_rows_multi(ctypes.byref(batch), arr, len(taus), _ptr(lp0), _ptr(lq),
                                   _ptr(entropy), _ptr(status), _ptr(workspace), ws_bytes,
                                   _stream(stream, workspace))
    if check and st != PS_OK:
        raise PsError(st, "ps_score_rows_multi")
    return st


def ps_selftest_wait_timeout(limit_ns: int, status: torch.Tensor, stream=None,
                             check: bool = True) -> int:
    """Diagnostic: a device wait that nothing completes gives up after limit_ns
    and sets PS_DEV_TIMEOUT in status (see include/ps.h)."""
    _need(status, torch.int32, "status")
    st = lib().ps_selftest_wait_timeout(int(limit_ns), _ptr(status), _stream(stream, status))
    if check and st != PS_OK:
        raise PsError(st, "ps_selftest_wait_timeout")
    return st


def ps_selftest_read(data: torch.Tensor, sink: torch.Tensor, stream=None,
                     check: bool = True) -> int:
    """Diagnostic: one plain streaming read of `data` (a contiguous device
    tensor, 16-byte aligned, a multiple of 16 bytes), folded into the int32
    `sink`; timing it gives the device's plain read rate (see include/ps.h)."""
    _need(sink, torch.int32, "sink")
    nbytes = data.numel() * data.element_size()
    st = lib().ps_selftest_read(_ptr(data), nbytes, _ptr(sink), _stream(stream, data))
    if check and st != PS_OK:
        raise PsError(st, "ps_selftest_read")
    return st


def ps_assemble_subtree(batch: PsSubtreeBatch, lp0: torch.Tensor, lq: torch.Tensor,
                        out: PsScoreOut, stream=None, check: bool = True) -> int:
    _need(lp0, torch.float64, "lp0")
    _need(lq, torch.float64, "lq")
    st = lib().ps_assemble_subtree(ctypes.byref(batch), _ptr(lp0), _ptr(lq), ctypes.byref(out),
                                   _stream(stream, lp0))
    if check and st != PS_OK:
        raise PsError(st, "ps_assemble_subtree")
    return st


def ps_walk_subtree(tree: PsTree, log_accept: torch.Tensor, out: PsWalkOut, stream=None,
                    check: bool = True) -> int:
    _need(log_accept, torch.float64, "log_accept")
    st = lib().ps_walk_subtree(ctypes.byref(tree), _ptr(log_accept), ctypes.byref(out),
                               _stream(stream, log_accept))
    if check and st != PS_OK:
        raise PsError(st, "ps_walk_subtree")
    return st


def ps_score_walk_subtree(batch: PsSubtreeBatch, tree: PsTree, out: PsScoreOut,
                          wout: PsWalkOut, workspace: torch.Tensor, stream=None,
                          check: bool = True) -> int:
    """Score, sum and walk one batch in one call (see include/ps.h)."""
    ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = lib().ps_score_walk_subtree(ctypes.byref(batch), ctypes.byref(tree), ctypes.byref(out),
                                     ctypes.byref(wout), ws_ptr, ws_bytes,
                                     _stream(stream, workspace))
    if check and st != PS_OK:
        raise PsError(st, "ps_score_walk_subtree")
    return st


def ps_carry_state(batch: PsSubtreeBatch, io: PsCarryIo, stream=None, check: bool = True) -> int:
    """The reached state's per-position values for the next round (see
    include/ps.h)."""
    st = lib().ps_carry_state(ctypes.byref(batch), ctypes.byref(io), _stream(stream, None))
    if check and st != PS_OK:
        raise PsError(st, "ps_carry_state")
    return st


def make_carry_io(*, state_seg, row_lp0, row_lq, next_lp0, next_lq, status, row_entropy=None,
                  prev_lp0=None, prev_lq=None, prev_entropy=None, next_entropy=None,
                  loglik=None, confidence=None) -> PsCarryIo:
    io = PsCarryIo()
    _need(state_seg, torch.int32, "state_seg")
    _need(status, torch.int32, "status")
    io.state_seg, io.status = _ptr(state_seg), _ptr(status)
    for name, x, opt in (("row_lp0", row_lp0, False), ("row_lq", row_lq, False),
                         ("row_entropy", row_entropy, True), ("prev_lp0", prev_lp0, True),
                         ("prev_lq", prev_lq, True), ("prev_entropy", prev_entropy, True),
                         ("next_lp0", next_lp0, False), ("next_lq", next_lq, False),
                         ("next_entropy", next_entropy, True), ("loglik", loglik, True),
                         ("confidence", confidence, True)):
        _need(x, torch.float64, name, optional=opt)
        setattr(io, name, _ptr(x))
    io._keep = (state_seg, row_lp0, row_lq, row_entropy, prev_lp0, prev_lq, prev_entropy,
                next_lp0, next_lq, next_entropy, loglik, confidence, status)
    return io


def ps_build_bfs_tree(T: int, n_pf: int, depth_cap: int | None, cuts) -> dict:
    """BFS request collection for one chain (host; see include/ps.h)."""
    cuts = np.ascontiguousarray(cuts, dtype=np.int32)
    n_cuts = int(cuts.shape[0])
    max_nodes, max_seg = 1 + 2 * n_cuts, n_pf + 1
    arr = {k: np.empty(max_nodes, np.int32) for k in ("acc", "rej", "req", "node_cut",
                                                      "deferred_cut")}
    seg = {k: np.empty(max_seg, np.int32) for k in ("seg_cut", "seg_src")}
    nn, ns, used = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = lib().ps_build_bfs_tree(int(T), int(n_pf), -1 if depth_cap is None else int(depth_cap),
                                 cuts.ctypes.data if n_cuts else None, n_cuts, max_nodes,
                                 max_seg, arr["acc"].ctypes.data, arr["rej"].ctypes.data,
                                 arr["req"].ctypes.data, arr["node_cut"].ctypes.data,
                                 arr["deferred_cut"].ctypes.data, seg["seg_cut"].ctypes.data,
                                 seg["seg_src"].ctypes.data, ctypes.byref(nn), ctypes.byref(ns),
                                 ctypes.byref(used))
    if st != PS_OK:
        raise PsError(st, "ps_build_bfs_tree")
    out = {k: v[:nn.value].copy() for k, v in arr.items()}
    out.update({k: v[:ns.value].copy() for k, v in seg.items()})
    out["cuts_used"] = used.value
    return out


def ps_predictive_allocation(acc, rej, candidate, h_acc, budget: int) -> tuple[float, np.ndarray]:
    """The eq. (19) dynamic program (host; see include/ps.h)."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    rej = np.ascontiguousarray(rej, dtype=np.int32)
    cand = np.ascontiguousarray(candidate, dtype=np.uint8)
    h = np.ascontiguousarray(h_acc, dtype=np.float64)
    n = int(acc.shape[0])
    sel = np.zeros(n, np.uint8)
    val = ctypes.c_double()
    st = lib().ps_predictive_allocation(n, acc.ctypes.data, rej.ctypes.data, cand.ctypes.data,
                                        h.ctypes.data, int(budget), ctypes.byref(val),
                                        sel.ctypes.data)
    if st != PS_OK:
        raise PsError(st, "ps_predictive_allocation")
    return val.value, sel.astype(bool)


def ps_midpoint_branch_probability(p_accept: float, p_reject: float) -> float:
    return float(lib().ps_midpoint_branch_probability(float(p_accept), float(p_reject)))


def ps_validate_subtree(batch: PsSubtreeBatch | None, tree: PsTree | None) -> tuple[int, str]:
    buf = ctypes.create_string_buffer(256)
    st = lib().ps_validate_subtree(ctypes.byref(batch) if batch is not None else None,
                                   ctypes.byref(tree) if tree is not None else None, buf, 256)
    return int(st), buf.value.decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError("tensors passed to libps must be contiguous")
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        if not x.flags.c_contiguous:
            raise ValueError("arrays passed to libps must be C-contiguous")
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(stream, like: torch.Tensor | None):
    if stream is None:
        dev = like.device if like is not None else None
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_NP_OF = {torch.int32: np.int32, torch.int64: np.int64, torch.float64: np.float64,
          torch.int8: np.int8}


def _need(x, dtype: torch.dtype, name: str, optional: bool = False):
    if x is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if isinstance(x, torch.Tensor):
        if x.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    elif isinstance(x, np.ndarray):
        if x.dtype != _NP_OF[dtype]:
            raise TypeError(f"{name} must be {_NP_OF[dtype]}, got {x.dtype}")
    else:
        raise TypeError(f"{name}: tensor or ndarray expected")


def make_batch(*, V: int, T: int, alpha: float, tau: float, chain_seg0, seg_row0, seg_cut,
               seg_src, logits=None, tokens=None, row_index=None, n_rows: int | None = None,
               n_logit_rows: int | None = None, ld: int | None = None,
               dtype: int | None = None, eps: float = 0.01, root_lp0=None,
               root_lq=None, flags: int = 0) -> PsSubtreeBatch:
    """Fill a ps_subtree_batch from tensors (device for scoring, host for validation)."""
    _need(chain_seg0, torch.int32, "chain_seg0")
    _need(seg_row0, torch.int64, "seg_row0")
    _need(seg_cut, torch.int32, "seg_cut")
    _need(seg_src, torch.int32, "seg_src")
    _need(tokens, torch.int32, "tokens", optional=True)
    _need(row_index, torch.int64, "row_index", optional=True)
    _need(root_lp0, torch.float64, "root_lp0", optional=True)
    _need(root_lq, torch.float64, "root_lq", optional=True)
    b = PsSubtreeBatch()
    b.V, b.T = int(V), int(T)
    b.n_chains = int(chain_seg0.shape[0]) - 1
    b.n_seg = int(seg_cut.shape[0])
    b.flags = int(flags)
    if n_rows is None:
        n_rows = int(tokens.shape[0]) if tokens is not None else 0
    b.n_rows = int(n_rows)
    if logits is not None:
        if dtype is None:
            if logits.dtype == torch.bfloat16:
                dtype = PS_BF16
            elif logits.dtype == torch.float32:
                dtype = PS_F32
            else:
                raise TypeError(f"logits must be bf16 or f32, got {logits.dtype}")
        if ld is None:
            ld = int(logits.shape[-1])
        if n_logit_rows is None:
            n_logit_rows = int(logits.shape[0])
    b.dtype = int(PS_BF16 if dtype is None else dtype)
    if ld is None:                       # host-only validation: smallest legal stride
        per16 = 8 if b.dtype == PS_BF16 else 4
        ld = -(-int(V) // per16) * per16
    b.ld = int(ld)
    b.n_logit_rows = int(0 if n_logit_rows is None else n_logit_rows)
    b.alpha, b.tau, b.eps = float(alpha), float(tau), float(eps)
    b.chain_seg0, b.seg_row0 = _ptr(chain_seg0), _ptr(seg_row0)
    b.seg_cut, b.seg_src = _ptr(seg_cut), _ptr(seg_src)
    b.logits, b.row_index, b.tokens = _ptr(logits), _ptr(row_index), _ptr(tokens)
    b.root_lp0, b.root_lq = _ptr(root_lp0), _ptr(root_lq)
    b._keep = (chain_seg0, seg_row0, seg_cut, seg_src, logits, tokens, row_index, root_lp0,
               root_lq)
    return b


def make_score_out(*, log_accept, status, lp0=None, lq=None, lp_y=None, lq_y=None, lp_x=None,
                   lq_x=None, log_ratio=None, entropy=None, eps_class=None) -> PsScoreOut:
    o = PsScoreOut()
    for name, x in (("lp0", lp0), ("lq", lq), ("lp_y", lp_y), ("lq_y", lq_y), ("lp_x", lp_x),
                    ("lq_x", lq_x), ("log_ratio", log_ratio), ("log_accept", log_accept),
                    ("entropy", entropy)):
        _need(x, torch.float64, name, optional=name != "log_accept")
        setattr(o, name, _ptr(x))
    _need(status, torch.int32, "status")
    _need(eps_class, torch.int8, "eps_class", optional=True)
    o.status = _ptr(status)
    o.eps_class = _ptr(eps_class)
    o._keep = (lp0, lq, lp_y, lq_y, lp_x, lq_x, log_ratio, log_accept, status, entropy,
               eps_class)
    return o


def make_tree(*, chain_node0, chain_seg0, acc, rej, req, u, max_steps: int) -> PsTree:
    for name, x in (("chain_node0", chain_node0), ("chain_seg0", chain_seg0), ("acc", acc),
                    ("rej", rej), ("req", req)):
        _need(x, torch.int32, name)
    _need(u, torch.float64, "u")
    t = PsTree()
    t.n_chains = int(chain_node0.shape[0]) - 1
    t.n_nodes = int(acc.shape[0])
    t.n_seg = int(u.shape[0])
    t.max_steps = int(max_steps)
    t.chain_node0, t.chain_seg0 = _ptr(chain_node0), _ptr(chain_seg0)
    t.acc, t.rej, t.req, t.u = _ptr(acc), _ptr(rej), _ptr(req), _ptr(u)
    t._keep = (chain_node0, chain_seg0, acc, rej, req, u)
    return t


def make_walk_out(*, state_seg, end_node, k_delta, status, path=None) -> PsWalkOut:
    o = PsWalkOut()
    for name, x in (("state_seg", state_seg), ("end_node", end_node), ("k_delta", k_delta),
                    ("status", status)):
        _need(x, torch.int32, name)
        setattr(o, name, _ptr(x))
    _need(path, torch.int32, "path", optional=True)
    o.path = _ptr(path)
    o._keep = (state_seg, end_node, k_delta, status, path)
    return o


def dev_status_names(bits: int) -> list[str]:
    return [n for b, n in PS_DEV_BITS.items() if bits & b]


@dataclass
class DeviceSubtree:
    """A subtree batch resident on one GPU, with its outputs and workspace.

    Built from host arrays of the layout (chain_seg0, seg_row0, seg_cut,
    seg_src, chain_node0, acc, rej, req), the acceptance uniforms and the
    device tensors of logits and tokens.
    """

    batch: PsSubtreeBatch
    tree: PsTree
    score_out: PsScoreOut
    walk_out: PsWalkOut
    workspace: torch.Tensor
    t: dict

    @classmethod
    def create(cls, *, layout, u, logits: torch.Tensor, tokens: torch.Tensor, V: int,
               alpha: float, tau: float, max_steps: int, row_index: torch.Tensor | None = None,
               per_row: bool = True, sums: bool = True, path: bool = True,
               entropy: bool = False, eps: float | None = None,
               root_lp0: torch.Tensor | None = None,
               root_lq: torch.Tensor | None = None, flags: int = 0) -> "DeviceSubtree":
        dev = logits.device
        i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
        t = dict(
            chain_seg0=i32(layout.chain_seg0),
            seg_row0=torch.as_tensor(np.ascontiguousarray(layout.seg_row0, dtype=np.int64)).to(dev),
            seg_cut=i32(layout.seg_cut), seg_src=i32(layout.seg_src),
            chain_node0=i32(layout.chain_node0), acc=i32(layout.acc), rej=i32(layout.rej),
            req=i32(layout.req),
            u=torch.as_tensor(np.ascontiguousarray(u, dtype=np.float64)).to(dev),
            logits=logits, tokens=tokens, row_index=row_index,
        )
        n_rows = int(layout.seg_row0[-1])
        n_seg = int(len(layout.seg_cut))
        n_chains = int(len(layout.chain_seg0)) - 1
        f64 = lambda n: torch.empty(n, dtype=torch.float64, device=dev)
        t["lp0"] = f64(n_rows) if per_row else None
        t["lq"] = f64(n_rows) if per_row else None
        for k in ("lp_y", "lq_y", "lp_x", "lq_x", "log_ratio"):
            t[k] = f64(n_seg) if sums else None
        t["log_accept"] = f64(n_seg)
        t["entropy"] = f64(n_rows) if entropy else None
        t["eps_class"] = (torch.empty(n_seg, dtype=torch.int8, device=dev)
                          if eps is not None else None)
        t["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        t["wstatus"] = torch.zeros(1, dtype=torch.int32, device=dev)
        for k in ("state_seg", "end_node", "k_delta"):
            t[k] = torch.empty(n_chains, dtype=torch.int32, device=dev)
        t["path"] = (torch.empty(n_chains * (max_steps + 1), dtype=torch.int32, device=dev)
                     if path else None)
        batch = make_batch(V=V, T=layout.T, alpha=alpha, tau=tau, chain_seg0=t["chain_seg0"],
                           seg_row0=t["seg_row0"], seg_cut=t["seg_cut"], seg_src=t["seg_src"],
                           logits=logits, tokens=tokens, row_index=row_index, n_rows=n_rows,
                           eps=0.01 if eps is None else eps, root_lp0=root_lp0,
                           root_lq=root_lq, flags=flags)
        ws_bytes = ps_score_workspace_bytes(batch)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        sout = make_score_out(log_accept=t["log_accept"], status=t["status"], lp0=t["lp0"],
                              lq=t["lq"], lp_y=t["lp_y"], lq_y=t["lq_y"], lp_x=t["lp_x"],
                              lq_x=t["lq_x"], log_ratio=t["log_ratio"], entropy=t["entropy"],
                              eps_class=t["eps_class"])
        tree = make_tree(chain_node0=t["chain_node0"], chain_seg0=t["chain_seg0"], acc=t["acc"],
                         rej=t["rej"], req=t["req"], u=t["u"], max_steps=max_steps)
        wout = make_walk_out(state_seg=t["state_seg"], end_node=t["end_node"],
                             k_delta=t["k_delta"], status=t["wstatus"], path=t["path"])
        return cls(batch=batch, tree=tree, score_out=sout, walk_out=wout, workspace=ws, t=t)

    def score(self, stream=None) -> None:
        ps_score_subtree(self.batch, self.score_out, self.workspace, stream)

    def score_rows(self, stream=None) -> None:
        """First half of score(): per-row log-probabilities into t['lp0'], t['lq']."""
        ps_score_rows(self.batch, self.t["lp0"], self.t["lq"], self.t["status"],
                      self.workspace, stream, entropy=self.t["entropy"])

    def assemble(self, stream=None) -> None:
        """Second half of score(): suffix sums and log A from t['lp0'], t['lq']."""
        ps_assemble_subtree(self.batch, self.t["lp0"], self.t["lq"], self.score_out, stream)

    def walk(self, stream=None) -> None:
        ps_walk_subtree(self.tree, self.t["log_accept"], self.walk_out, stream)

    def step(self, stream=None, fused: bool = True) -> None:
        """One pass of the whole path: score, sum and walk in one call
        (ps_score_walk_subtree), or with fused=False in two
        (ps_score_subtree, then ps_walk_subtree)."""
        if fused:
            ps_score_walk_subtree(self.batch, self.tree, self.score_out, self.walk_out,
                                  self.workspace, stream)
        else:
            self.score(stream)
            self.walk(stream)

    def carry(self, prev: dict | None = None, stream=None) -> dict:
        """Per-position values of each chain's reached state for the next
        round (after step()); prev holds the current state's values for the
        positions below the root cut ("lp0", "lq" and optionally "entropy",
        each [n_chains, T])."""
        t = self.t
        n_chains = int(t["chain_seg0"].shape[0]) - 1
        T = int(self.batch.T)
        dev = t["log_accept"].device
        out = {k: torch.empty((n_chains, T), dtype=torch.float64, device=dev)
               for k in ("lp0", "lq")}
        ent = t.get("entropy") is not None
        if ent:
            out["entropy"] = torch.empty((n_chains, T), dtype=torch.float64, device=dev)
        out["loglik"] = torch.empty(n_chains, dtype=torch.float64, device=dev)
        if ent:
            out["confidence"] = torch.empty(n_chains, dtype=torch.float64, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        prev = prev or {}
        io = make_carry_io(state_seg=t["state_seg"], row_lp0=t["lp0"], row_lq=t["lq"],
                           row_entropy=t.get("entropy"), prev_lp0=prev.get("lp0"),
                           prev_lq=prev.get("lq"), prev_entropy=prev.get("entropy"),
                           next_lp0=out["lp0"], next_lq=out["lq"],
                           next_entropy=out.get("entropy"), loglik=out["loglik"],
                           confidence=out.get("confidence"), status=status)
        ps_carry_state(self.batch, io, stream)
        out["status"] = status
        return out
