"""ctypes binding of libssmtree (include/ssm_tree.h), same names as the C ABI.

Argument marshalling only: each wrapper checks that the torch tensors it is
given have the dtype, device, contiguity and element count the C signature
expects (the C side sees bare pointers and cannot), then calls the library on
the current CUDA stream (or the one passed).  All arithmetic runs in the
library's CUDA kernels; there is no fallback: if libssmtree.so is not built,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

from . import build as _build

SSM_OK = 0
SSM_ERR_INVALID_ARG = -1
SSM_ERR_BAD_TREE = -2
SSM_ERR_CAPACITY = -3
SSM_ERR_CUDA = -4
SSM_ERR_RANGE = -5
SSM_STATUS_BAD_LAYOUT = 1
SSM_STATUS_PATH_RANGE = 2
SSM_STATUS_K_RANGE = 4
SSM_STATUS_WALK_TRUNCATED = 8
SSM_STATUS_TIMEOUT = 16
SSM_MAX_NODES = 64
SSM_MAX_DEPTH = 15
SSM_MAX_PATH = 256
SSM_MAX_CHAIN_NODES = 4096
SSM_NOALLOC_WORKSPACE_BYTES = 16 << 20
NODE_WORDS = 8  # int32 words per ssm_node record


class SSMError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class ssm_dims(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("d_state", ctypes.c_int32),
                ("conv_width", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("ring_cap", ctypes.c_int32)]


class ssm_params(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("A_log", ctypes.c_void_p), ("D", ctypes.c_void_p)]


@dataclass(frozen=True)
class Dims:
    n_heads: int
    n_layers: int = 1
    ring_cap: int = 20
    head_dim: int = 64
    d_state: int = 128
    conv_width: int = 4

    @property
    def d_inner(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def conv_dim(self) -> int:
        return self.d_inner + 2 * self.d_state

    def c(self) -> ssm_dims:
        return ssm_dims(self.n_heads, self.head_dim, self.d_state, self.conv_width, self.n_layers, self.ring_cap)


_LIB = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "ssm_version": (_I, []),
    "ssm_last_error": (ctypes.c_char_p, []),
    "ssm_tree_layout_build": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P]),
    "ssm_tree_verify": (ctypes.c_int, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "ssm_tree_verify_workspace_size": (ctypes.c_size_t, [_P, _I, _I, _I]),
    "ssm_tree_verify_noalloc": (ctypes.c_int, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ssm_accept_path": (ctypes.c_int, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ssm_commit": (ctypes.c_int, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ssm_commit_verify_workspace_size": (ctypes.c_size_t, [_P, _I, _I, _I, _I]),
    "ssm_commit_verify": (ctypes.c_int, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                         _P, ctypes.c_size_t, _P, _P]),
    "ssm_commit_verify_prep": (ctypes.c_int, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P,
                                              _P, _P, ctypes.c_size_t, _P, _P]),
    "ssm_commit_verify_main": (ctypes.c_int, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P,
                                              _P, _P, ctypes.c_size_t, _P, _P]),
    "ssm_draft_step": (ctypes.c_int, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ssm_replay": (ctypes.c_int, [_P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ssm_draft_tree_level": (ctypes.c_int, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                            ctypes.c_size_t, _P, _P]),
    "ssm_draft_tree_workspace_size": (ctypes.c_size_t, [_P, _I, _I]),
    "ssm_selftest_bounded_wait": (ctypes.c_int, [_I, _P, _P]),
    "ssm_set_tuning": (ctypes.c_int, [ctypes.c_char_p, _I]),
    "ssm_selftest_silu": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P]),
    "ssm_draft_tree_commit": (ctypes.c_int, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
}


def library_path() -> str:
    return _build.lib_path()


def lib():
    """The loaded libssmtree (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libssmtree is not built ({path} missing): run "
                               "`python -m speculative_decoding_mamba2_gb300.build` or __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def ssm_version() -> int:
    return int(lib().ssm_version())


def ssm_last_error() -> str:
    return lib().ssm_last_error().decode()


def _check(rc: int):
    if rc != SSM_OK:
        raise SSMError(rc, ssm_last_error())


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _dev(t: torch.Tensor, name: str, dtype, numel: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
    return ctypes.c_void_p(t.data_ptr())


def _ptr(t: torch.Tensor, name: str, dtype, numel: int):
    """Integer address (for ctypes struct fields)."""
    return _dev(t, name, dtype, numel).value


def _opt_status(status):
    return None if status is None else _dev(status, "status", torch.int32, 1)


def _stream(stream, like: torch.Tensor):
    if stream is None:
        stream = torch.cuda.current_stream(like.device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _params(prm: dict, d: Dims, layers: int) -> ssm_params:
    return ssm_params(_ptr(prm["conv_w"], "conv_w", torch.float32, layers * d.conv_dim * d.conv_width),
                      _ptr(prm["conv_b"], "conv_b", torch.float32, layers * d.conv_dim),
                      _ptr(prm["dt_bias"], "dt_bias", torch.float32, layers * d.n_heads),
                      _ptr(prm["A_log"], "A_log", torch.float32, layers * d.n_heads),
                      _ptr(prm["D"], "D", torch.float32, layers * d.n_heads))


# ---------------------------------------------------------------------------
# the C ABI, one wrapper per entry point
# ---------------------------------------------------------------------------
def ssm_tree_layout_build(parent, max_branches: int = 0, max_depth: int = 0):
    """Host call.  parent: int array [n_seq][n] (or [n]).  Returns (layout int32
    [n_seq][n][8] = ssm_node records, deepest depth)."""
    par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    if par.ndim == 1:
        par = par[None]
    if par.ndim != 2 or par.shape[1] < 1:
        raise ValueError("parent must be [n_seq][n_nodes]")
    S, n = par.shape
    out = np.zeros((S, n, NODE_WORDS), np.int32)
    depth = ctypes.c_int32(0)
    _check(lib().ssm_tree_layout_build(par.ctypes.data_as(_P), S, n, int(max_branches), int(max_depth),
                                       out.ctypes.data_as(_P), ctypes.byref(depth)))
    return out, int(depth.value)


def ssm_tree_verify_workspace_size(dims: Dims, n_seq: int, n_nodes: int, max_depth: int) -> int:
    """Bytes of device workspace ssm_tree_verify needs (host call)."""
    cd = dims.c()
    b = lib().ssm_tree_verify_workspace_size(ctypes.byref(cd), n_seq, n_nodes, max_depth)
    if b == 0:
        raise SSMError(SSM_ERR_CAPACITY, ssm_last_error())
    return int(b)


def ssm_tree_verify(dims: Dims, params: dict, n_seq: int, n_nodes: int, max_depth: int, layout, xBC, dt, h0, ring,
                    ring_head, y, workspace, status=None, stream=None):
    d, I, n = dims, n_seq * dims.n_layers, n_nodes
    cd = d.c()
    cp = _params(params, d, d.n_layers)
    _check(lib().ssm_tree_verify(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, n, max_depth,
        _dev(layout, "layout", torch.int32, n_seq * n * NODE_WORDS),
        _dev(xBC, "xBC", torch.bfloat16, I * n * d.conv_dim), _dev(dt, "dt", torch.bfloat16, I * n * d.n_heads),
        _dev(h0, "h0", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
        _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim),
        _dev(ring_head, "ring_head", torch.int32, I), _dev(y, "y", torch.float32, I * n * d.d_inner),
        _dev(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _opt_status(status), _stream(stream, h0)))


def ssm_tree_verify_noalloc(dims: Dims, params: dict, n_seq: int, n_nodes: int, max_depth: int, layout, xBC, dt, h0,
                            ring, ring_head, y, status=None, stream=None):
    """ssm_tree_verify for callers that cannot allocate device memory: the scratch
    is the library's own SSM_NOALLOC_WORKSPACE_BYTES array (shared by every call;
    overlapping calls race).  Batches needing more raise SSMError(SSM_ERR_CAPACITY).
    The call runs with h0's device current, so the library looks up that device's array."""
    d, I, n = dims, n_seq * dims.n_layers, n_nodes
    cd = d.c()
    cp = _params(params, d, d.n_layers)
    if not isinstance(h0, torch.Tensor) or not h0.is_cuda:
        raise ValueError("h0: must be a CUDA tensor")
    with torch.cuda.device(h0.device):
        _check(lib().ssm_tree_verify_noalloc(
            ctypes.byref(cd), ctypes.byref(cp), n_seq, n, max_depth,
            _dev(layout, "layout", torch.int32, n_seq * n * NODE_WORDS),
            _dev(xBC, "xBC", torch.bfloat16, I * n * d.conv_dim), _dev(dt, "dt", torch.bfloat16, I * n * d.n_heads),
            _dev(h0, "h0", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
            _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim),
            _dev(ring_head, "ring_head", torch.int32, I), _dev(y, "y", torch.float32, I * n * d.d_inner),
            _opt_status(status), _stream(stream, h0)))


def ssm_accept_path(n_seq: int, n_nodes: int, max_path: int, layout, tok, tgt, path, path_len, bonus, status=None,
                    stream=None):
    S, n = n_seq, n_nodes
    _check(lib().ssm_accept_path(
        S, n, max_path, _dev(layout, "layout", torch.int32, S * n * NODE_WORDS),
        _dev(tok, "tok", torch.int32, S * n), _dev(tgt, "tgt", torch.int32, S * n),
        _dev(path, "path", torch.int32, S * max_path), _dev(path_len, "path_len", torch.int32, S),
        _dev(bonus, "bonus", torch.int32, S), _opt_status(status), _stream(stream, tok)))


def ssm_commit(dims: Dims, params: dict, n_seq: int, n_nodes: int, layout, max_path: int, path, path_len, xBC, dt, h,
               ring, ring_head, status=None, stream=None):
    d, I, n = dims, n_seq * dims.n_layers, n_nodes
    cd = d.c()
    cp = _params(params, d, d.n_layers)
    _check(lib().ssm_commit(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, n, _dev(layout, "layout", torch.int32, n_seq * n * NODE_WORDS),
        max_path, _dev(path, "path", torch.int32, n_seq * max_path), _dev(path_len, "path_len", torch.int32, n_seq),
        _dev(xBC, "xBC", torch.bfloat16, I * n * d.conv_dim), _dev(dt, "dt", torch.bfloat16, I * n * d.n_heads),
        _dev(h, "h", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
        _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim),
        _dev(ring_head, "ring_head", torch.int32, I), _opt_status(status), _stream(stream, h)))


def ssm_commit_verify_workspace_size(dims: Dims, n_seq: int, n_nodes: int, max_depth: int, prev_max_path: int) -> int:
    cd = dims.c()
    b = lib().ssm_commit_verify_workspace_size(ctypes.byref(cd), n_seq, n_nodes, max_depth, prev_max_path)
    if b == 0:
        raise SSMError(SSM_ERR_CAPACITY, ssm_last_error())
    return int(b)


def ssm_commit_verify(dims: Dims, params: dict, n_seq: int, prev_n_nodes: int, prev_layout, prev_max_path: int,
                      prev_path, prev_path_len, prev_xBC, prev_dt, n_nodes: int, max_depth: int, layout, xBC, dt, h,
                      ring, ring_head, y, workspace, status=None, stream=None, part: str = "all"):
    """ssm_commit of the previous tree's accepted path, then ssm_tree_verify of the
    next tree from the committed state, with one read and one write of h.
    part="prep" / "main" issues only one half (ssm_commit_verify_prep / _main): the
    prep needs only the tree's B|C channels and dt, the main the x channels too."""
    d, I, n, pn = dims, n_seq * dims.n_layers, n_nodes, prev_n_nodes
    cd = d.c()
    cp = _params(params, d, d.n_layers)
    entry = {"all": "ssm_commit_verify", "prep": "ssm_commit_verify_prep", "main": "ssm_commit_verify_main"}[part]
    _check(getattr(lib(), entry)(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, pn,
        _dev(prev_layout, "prev_layout", torch.int32, n_seq * pn * NODE_WORDS), prev_max_path,
        _dev(prev_path, "prev_path", torch.int32, n_seq * prev_max_path),
        _dev(prev_path_len, "prev_path_len", torch.int32, n_seq),
        _dev(prev_xBC, "prev_xBC", torch.bfloat16, I * pn * d.conv_dim),
        _dev(prev_dt, "prev_dt", torch.bfloat16, I * pn * d.n_heads),
        n, max_depth, _dev(layout, "layout", torch.int32, n_seq * n * NODE_WORDS),
        _dev(xBC, "xBC", torch.bfloat16, I * n * d.conv_dim), _dev(dt, "dt", torch.bfloat16, I * n * d.n_heads),
        _dev(h, "h", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
        _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim),
        _dev(ring_head, "ring_head", torch.int32, I), _dev(y, "y", torch.float32, I * n * d.d_inner),
        _dev(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _opt_status(status), _stream(stream, h)))


def ssm_draft_step(dims: Dims, params: dict, n_seq: int, step: int, log_cap: int, xBC_t, dt_t, h_in, h_out, ring,
                   ring_head, log_delta, log_B, log_x, log_len, y, status=None, stream=None):
    d, I = dims, n_seq * dims.n_layers
    cd = d.c()
    cp = _params(params, d, d.n_layers)
    S = I * d.n_heads * d.head_dim * d.d_state
    _check(lib().ssm_draft_step(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, step, log_cap,
        _dev(xBC_t, "xBC_t", torch.bfloat16, I * d.conv_dim), _dev(dt_t, "dt_t", torch.bfloat16, I * d.n_heads),
        _dev(h_in, "h_in", torch.float32, S), _dev(h_out, "h_out", torch.float32, S),
        _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim),
        _dev(ring_head, "ring_head", torch.int32, I),
        _dev(log_delta, "log_delta", torch.float32, I * log_cap * d.n_heads),
        _dev(log_B, "log_B", torch.float32, I * log_cap * d.d_state),
        _dev(log_x, "log_x", torch.float32, I * log_cap * d.d_inner), _dev(log_len, "log_len", torch.int32, I),
        _dev(y, "y", torch.float32, I * d.d_inner), _opt_status(status), _stream(stream, h_out)))


def ssm_replay(dims: Dims, params: dict, n_seq: int, log_cap: int, k, log_delta, log_B, log_x, log_len, h_ckpt,
               ring_head, status=None, stream=None):
    d, I = dims, n_seq * dims.n_layers
    cd = d.c()
    cp = ssm_params(None, None, None, _ptr(params["A_log"], "A_log", torch.float32, d.n_layers * d.n_heads), None)
    _check(lib().ssm_replay(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, log_cap, _dev(k, "k", torch.int32, n_seq),
        _dev(log_delta, "log_delta", torch.float32, I * log_cap * d.n_heads),
        _dev(log_B, "log_B", torch.float32, I * log_cap * d.d_state),
        _dev(log_x, "log_x", torch.float32, I * log_cap * d.d_inner), _dev(log_len, "log_len", torch.int32, I),
        _dev(h_ckpt, "h_ckpt", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
        _dev(ring_head, "ring_head", torch.int32, I), _opt_status(status), _stream(stream, h_ckpt)))


def ssm_draft_tree_workspace_size(dims: Dims, n_seq: int, n_nodes: int) -> int:
    """Bytes of device workspace ssm_draft_tree_level needs (host call)."""
    cd = dims.c()
    b = lib().ssm_draft_tree_workspace_size(ctypes.byref(cd), n_seq, n_nodes)
    if b == 0:
        raise SSMError(SSM_ERR_INVALID_ARG, ssm_last_error())
    return int(b)


def ssm_draft_tree_level(dims: Dims, params: dict, n_seq: int, n_nodes: int, level: int, layout, xBC, dt, h_ckpt,
                         ring, ring_head, log_delta, log_B, log_x, y, workspace, status=None, stream=None):
    """One depth level of the draft tree: y and log rows of the nodes of depth `level`."""
    d, I, n = dims, n_seq * dims.n_layers, n_nodes
    cd = d.c()
    cp = _params(params, d, d.n_layers)
    _check(lib().ssm_draft_tree_level(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, n, level,
        _dev(layout, "layout", torch.int32, n_seq * n * NODE_WORDS),
        _dev(xBC, "xBC", torch.bfloat16, I * n * d.conv_dim), _dev(dt, "dt", torch.bfloat16, I * n * d.n_heads),
        _dev(h_ckpt, "h_ckpt", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
        _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim), _dev(ring_head, "ring_head", torch.int32, I),
        _dev(log_delta, "log_delta", torch.float32, I * n * d.n_heads),
        _dev(log_B, "log_B", torch.float32, I * n * d.d_state),
        _dev(log_x, "log_x", torch.float32, I * n * d.d_inner),
        _dev(y, "y", torch.float32, I * n * d.d_inner), _dev(workspace, "workspace", torch.uint8),
        ctypes.c_size_t(workspace.numel()), _opt_status(status), _stream(stream, y)))


def ssm_draft_tree_commit(dims: Dims, params: dict, n_seq: int, n_nodes: int, layout, max_path: int, path, path_len,
                          log_delta, log_B, log_x, xBC, h_ckpt, ring, ring_head, status=None, stream=None):
    """The accepted path's logged updates into h_ckpt, its rows into the ring, head += path_len."""
    d, I, n = dims, n_seq * dims.n_layers, n_nodes
    cd = d.c()
    cp = ssm_params(None, None, None, _ptr(params["A_log"], "A_log", torch.float32, d.n_layers * d.n_heads), None)
    _check(lib().ssm_draft_tree_commit(
        ctypes.byref(cd), ctypes.byref(cp), n_seq, n, _dev(layout, "layout", torch.int32, n_seq * n * NODE_WORDS),
        max_path, _dev(path, "path", torch.int32, n_seq * max_path), _dev(path_len, "path_len", torch.int32, n_seq),
        _dev(log_delta, "log_delta", torch.float32, I * n * d.n_heads),
        _dev(log_B, "log_B", torch.float32, I * n * d.d_state),
        _dev(log_x, "log_x", torch.float32, I * n * d.d_inner),
        _dev(xBC, "xBC", torch.bfloat16, I * n * d.conv_dim),
        _dev(h_ckpt, "h_ckpt", torch.float32, I * d.n_heads * d.head_dim * d.d_state),
        _dev(ring, "ring", torch.bfloat16, I * d.ring_cap * d.conv_dim),
        _dev(ring_head, "ring_head", torch.int32, I), _opt_status(status), _stream(stream, h_ckpt)))


def ssm_selftest_silu(v, out=None, stream=None):
    """The kernels' three SiLU forms on the fp32 CUDA tensor v: returns out [3, n]
    (FMA-pipe polynomial form, special-function form, expf form)."""
    n = v.numel()
    if out is None:
        out = torch.empty((3, n), dtype=torch.float32, device=v.device)
    _check(lib().ssm_selftest_silu(_dev(v, "v", torch.float32, n), _dev(out, "out", torch.float32, 3 * n), n,
                                   _stream(stream, v)))
    return out


def ssm_set_tuning(name: str, value: int):
    """Set a process-wide launch-plan override (0 = automatic); see include/ssm_tree.h."""
    _check(lib().ssm_set_tuning(name.encode(), int(value)))


def ssm_selftest_bounded_wait(limit_us: int, status, stream=None):
    """Run the library's bounded mbarrier wait on a barrier nothing arrives at (it gives up
    after limit_us and sets SSM_STATUS_TIMEOUT in `status`)."""
    _check(lib().ssm_selftest_bounded_wait(int(limit_us), _dev(status, "status", torch.int32, 1),
                                           _stream(stream, status)))


# ---------------------------------------------------------------------------
# the block's dense steps (include/ssm_layer.h)
# ---------------------------------------------------------------------------
class ssm_out_segment(ctypes.Structure):
    _fields_ = [("col", ctypes.c_int32), ("f32", ctypes.c_int32), ("ld", ctypes.c_int64), ("ptr", ctypes.c_void_p)]


_SIGS.update({
    "ssm_linear": (ctypes.c_int, [_I, _I, _I, _P, ctypes.c_int64, _P, ctypes.c_int64, _I, _P, _P, ctypes.c_int64, _P,
                                  _P]),
    "ssm_linear_tile_cols": (_I, []),
    "ssm_rmsnorm": (ctypes.c_int, [_I, _I, _P, ctypes.c_int64, _P, ctypes.c_float, _P, ctypes.c_int64, _P]),
    "ssm_gated_rmsnorm": (ctypes.c_int, [_I, _I, _P, ctypes.c_int64, _P, ctypes.c_int64, _P, ctypes.c_float, _P,
                                         ctypes.c_int64, _P]),
})


def _rows(t: torch.Tensor, name: str, dtype, cols: int | None = None):
    """A 2-D CUDA tensor whose rows are contiguous (any row stride): (pointer, rows, row stride)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError(f"{name}: must be 2-D with contiguous rows")
    if cols is not None and t.size(1) != cols:
        raise ValueError(f"{name}: {t.size(1)} columns, expected {cols}")
    return ctypes.c_void_p(t.data_ptr()), t.size(0), t.stride(0)


def ssm_linear_tile_cols() -> int:
    return int(lib().ssm_linear_tile_cols())


def ssm_linear(A, W, segments, residual=None, status=None, stream=None):
    """D = A · Wᵀ (+ residual) on the tensor cores.  A: bf16 [M, K], W: bf16 [N, K] (rows
    contiguous, any row stride).  segments: [(first column, out)], out a bf16 or fp32
    [M, width] view; the segments cover [0, N) in order.  residual: fp32 [M, N] or None
    (it may be the output itself)."""
    a, M, lda = _rows(A, "A", torch.bfloat16)
    w, N, ldw = _rows(W, "W", torch.bfloat16, A.size(1))
    K = A.size(1)
    segs = (ssm_out_segment * len(segments))()
    for i, (col, out) in enumerate(segments):
        end = segments[i + 1][0] if i + 1 < len(segments) else N
        p, rows, ld = _rows(out, f"segment {i}", out.dtype, end - col)
        if out.dtype not in (torch.bfloat16, torch.float32) or rows != M:
            raise ValueError(f"segment {i}: bf16 or fp32 with {M} rows")
        segs[i] = ssm_out_segment(col, 1 if out.dtype == torch.float32 else 0, ld, p.value)
    r, ldr = None, 0
    if residual is not None:
        r, rows, ldr = _rows(residual, "residual", torch.float32, N)
        if rows != M:
            raise ValueError("residual: M rows")
    _check(lib().ssm_linear(M, N, K, a, lda, w, ldw, len(segments), segs, r, ldr, _opt_status(status),
                            _stream(stream, A)))


def ssm_rmsnorm(x, w, eps: float, out, stream=None):
    """out (bf16) = w · x / sqrt(mean(x²) + eps) per row of x (fp32 [M, C])."""
    px, M, ldx = _rows(x, "x", torch.float32)
    C = x.size(1)
    po, Mo, ldo = _rows(out, "out", torch.bfloat16, C)
    if Mo != M:
        raise ValueError("out: M rows")
    _check(lib().ssm_rmsnorm(M, C, px, ldx, _dev(w, "w", torch.float32, C), float(eps), po, ldo, _stream(stream, x)))


def ssm_gated_rmsnorm(y, z, w, eps: float, out, stream=None):
    """out (bf16) = RMSNorm(y · SiLU(z)) · w per row; y fp32 [M, C], z bf16 [M, C]."""
    py, M, ldy = _rows(y, "y", torch.float32)
    C = y.size(1)
    pz, Mz, ldz = _rows(z, "z", torch.bfloat16, C)
    po, Mo, ldo = _rows(out, "out", torch.bfloat16, C)
    if Mz != M or Mo != M:
        raise ValueError("z, out: M rows")
    _check(lib().ssm_gated_rmsnorm(M, C, py, ldy, pz, ldz, _dev(w, "w", torch.float32, C), float(eps), po, ldo,
                                   _stream(stream, y)))
