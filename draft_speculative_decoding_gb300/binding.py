"""ctypes binding to libdfs.so, the C ABI declared in include/dfs.h.

Argument marshalling only: every step of the select-and-verify path runs in the
library's CUDA kernels. PyTorch supplies device memory and the current stream.
The functions carry the C names; outputs are allocated here with torch and
returned. A missing library is an error (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DFS_OK, DFS_ERR_INVALID, DFS_ERR_UNSUPPORTED, DFS_ERR_WORKSPACE, DFS_ERR_CUDA, DFS_ERR_TIMEOUT = \
    0, -1, -2, -3, -4, -5
DFS_BF16, DFS_FP32 = 0, 1
DFS_PATH_GREEDY, DFS_PATH_VITERBI, DFS_PATH_SAMPLE, DFS_PATH_SAMPLE_JOINT = 0, 1, 2, 3
K = 16

# Every symbol include/dfs.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int


class Dims(ctypes.Structure):
    _fields_ = [("B", _I), ("L", _I), ("K", _I), ("V", _I), ("d", _I), ("r", _I),
                ("dtype", _I), ("zdtype", _I)]


_DP = ctypes.POINTER(Dims)
SIGNATURES = {
    "dfs_version": ([], _I),
    "dfs_status_string": ([_I], ctypes.c_char_p),
    "dfs_workspace_size": ([_DP], ctypes.c_size_t),
    "dfs_set_trace_events": ([_P, _P], _I),
    "dfs_launch_count": ([], ctypes.c_uint64),
    "dfs_workspace_init": ([_P, ctypes.c_size_t, _P], _I),
    "dfs_get_device_error": ([_P, ctypes.c_size_t, ctypes.POINTER(_I), _P], _I),
    "dfs_lmhead_topk": ([_DP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
    "dfs_pair_score": ([_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
    "dfs_path_select": ([_DP, _P, _P, _I, _P, _P, _P], _I),
    "dfs_verify": ([_DP, _P, _P, ctypes.c_float, ctypes.c_uint64, _P, _P, _P, ctypes.c_size_t, _P],
                   _I),
    "dfs_verify_noalloc": ([_DP, _P, _P, ctypes.c_float, ctypes.c_uint64, _P, _P, _P], _I),
    "dfs_select_verify": ([_DP, _P, _P, _P, _P, _P, _P, _P, _I, ctypes.c_float, ctypes.c_uint64,
                           _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
    "dfs_quantize_rows_e4m3": ([_DP, _P, _P, _P, _P], _I),
    "dfs_e4m3_head_bytes": ([_I, _I], ctypes.c_size_t),
    "dfs_pack_e4m3_head": ([_I, _I, _P, _P, _P], _I),
    "dfs_lmhead_topk_e4m3": ([_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
    "dfs_select_verify_e4m3": ([_DP, _P, _P, _P, _P, _P, _P, _P, _P, _I, ctypes.c_float,
                                ctypes.c_uint64, _P, _P, _P, _P, _P, _P, _P, _P,
                                ctypes.c_size_t, _P], _I),
    "dfs_next_tokens": ([_I, _I, _P, _P, _P, _P], _I),
    "dfs_conv2tap_workspace_size": ([_I, _I, _I], ctypes.c_size_t),
    "dfs_conv2tap": ([_I, _I, _I, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
}

_lock = threading.Lock()
_lib = None


class DfsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libdfs.so (built in-tree by build.build()). Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = path or _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"libdfs.so not found at {path}; run "
                                   "draft_speculative_decoding_gb300.build.build() first")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().dfs_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != DFS_OK:
        raise DfsError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DFS_BF16
    if t.dtype == torch.float32:
        return DFS_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def make_dims(B, L, V, d, r, dtype: int, zdtype: int) -> Dims:
    return Dims(int(B), int(L), K, int(V), int(d), int(r), int(dtype), int(zdtype))


def dims_of(hidden: torch.Tensor, W: torch.Tensor, r: int, Z: torch.Tensor | None = None) -> Dims:
    B, L, d = hidden.shape
    V = W.shape[1]
    return make_dims(B, L, V, d, r, _code(hidden), _code(Z) if Z is not None else _code(hidden))


def dfs_workspace_size(dims: Dims) -> int:
    return int(load().dfs_workspace_size(ctypes.byref(dims)))


def alloc_workspace(dims: Dims, device=None, stream=None) -> torch.Tensor:
    """A zero-initialised workspace tensor for `dims` (uint8, 256-byte aligned by torch)."""
    n = dfs_workspace_size(dims)
    if n == 0:
        raise DfsError("dfs_workspace_size", DFS_ERR_UNSUPPORTED)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check("dfs_workspace_init", load().dfs_workspace_init(_ptr(ws), n, _stream(stream)))
    return ws


def dfs_set_trace_events(start=None, stop=None):
    """start/stop: torch.cuda.Event (created with enable_timing=True) or None. torch creates
    the underlying CUDA event on its first record(), so an unrecorded event is recorded once
    here to materialise it."""
    for ev in (start, stop):
        if ev is not None and not ev.cuda_event:
            ev.record()
    _check("dfs_set_trace_events", load().dfs_set_trace_events(
        None if start is None else ctypes.c_void_p(start.cuda_event),
        None if stop is None else ctypes.c_void_p(stop.cuda_event)))


def dfs_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().dfs_launch_count())


def dfs_get_device_error(ws: torch.Tensor, stream=None) -> int:
    err = _I(0)
    _check("dfs_get_device_error",
           load().dfs_get_device_error(_ptr(ws), ws.numel(), ctypes.byref(err), _stream(stream)))
    return err.value


def dfs_lmhead_topk(dims: Dims, hidden, W_vocab, ws, stream=None):
    P = dims.L - 1
    ids = torch.empty(dims.B, P, K, dtype=torch.int32, device=hidden.device)
    U = torch.empty(dims.B, P, K, dtype=torch.float32, device=hidden.device)
    _check("dfs_lmhead_topk", load().dfs_lmhead_topk(
        ctypes.byref(dims), _ptr(hidden), _ptr(W_vocab), _ptr(ids), _ptr(U), _ptr(ws), ws.numel(),
        _stream(stream)))
    return ids, U


def dfs_pair_score(dims: Dims, hidden, W_g, A, Btab, last_verified, cand_ids, cand_U, ws,
                   want_gate: bool = False, stream=None):
    P = dims.L - 1
    S = torch.empty(dims.B, P, K, K, dtype=torch.float32, device=hidden.device)
    gate = torch.empty(dims.B, P, dims.r, dtype=torch.float32, device=hidden.device) \
        if want_gate else None
    _check("dfs_pair_score", load().dfs_pair_score(
        ctypes.byref(dims), _ptr(hidden), _ptr(W_g), _ptr(A), _ptr(Btab), _ptr(last_verified),
        _ptr(cand_ids), _ptr(cand_U), _ptr(S), _ptr(gate), _ptr(ws), ws.numel(), _stream(stream)))
    return (S, gate) if want_gate else S


def dfs_path_select(dims: Dims, S, cand_ids, path_mode: int, stream=None):
    P = dims.L - 1
    path = torch.empty(dims.B, P, dtype=torch.int32, device=S.device)
    score = torch.empty(dims.B, dtype=torch.float32, device=S.device)
    _check("dfs_path_select", load().dfs_path_select(
        ctypes.byref(dims), _ptr(S), _ptr(cand_ids), int(path_mode), _ptr(path), _ptr(score),
        _stream(stream)))
    return path, score


def dfs_verify(dims: Dims, path, target_logits, temperature: float, seed: int, ws, stream=None):
    out = torch.empty(dims.B, dims.L, dtype=torch.int32, device=path.device)
    acc = torch.empty(dims.B, dtype=torch.int32, device=path.device)
    _check("dfs_verify", load().dfs_verify(
        ctypes.byref(dims), _ptr(path), _ptr(target_logits), float(temperature),
        int(seed) & (2**64 - 1), _ptr(out), _ptr(acc), _ptr(ws), ws.numel(), _stream(stream)))
    return out, acc


def dfs_verify_noalloc(dims: Dims, path, target_logits, temperature: float, seed: int,
                       stream=None):
    """dfs_verify with the library's built-in scratch: no workspace, nothing allocated by
    the library (the outputs below are allocated here, by the caller's side)."""
    out = torch.empty(dims.B, dims.L, dtype=torch.int32, device=path.device)
    acc = torch.empty(dims.B, dtype=torch.int32, device=path.device)
    _check("dfs_verify_noalloc", load().dfs_verify_noalloc(
        ctypes.byref(dims), _ptr(path), _ptr(target_logits), float(temperature),
        int(seed) & (2**64 - 1), _ptr(out), _ptr(acc), _stream(stream)))
    return out, acc


def dfs_select_verify(dims: Dims, hidden, W_vocab, W_g, A, Btab, last_verified, target_logits,
                      path_mode: int, temperature: float, seed: int, ws, *, outputs=None,
                      want_intermediates: bool = False, stream=None):
    """The fused step. `outputs` may pass preallocated (path, out_tokens, accept_len)."""
    P = dims.L - 1
    dev = hidden.device
    if outputs is None:
        outputs = (torch.empty(dims.B, P, dtype=torch.int32, device=dev),
                   torch.empty(dims.B, dims.L, dtype=torch.int32, device=dev),
                   torch.empty(dims.B, dtype=torch.int32, device=dev))
    path, out, acc = outputs
    ids = U = S = score = None
    if want_intermediates:
        ids = torch.empty(dims.B, P, K, dtype=torch.int32, device=dev)
        U = torch.empty(dims.B, P, K, dtype=torch.float32, device=dev)
        S = torch.empty(dims.B, P, K, K, dtype=torch.float32, device=dev)
        score = torch.empty(dims.B, dtype=torch.float32, device=dev)
    _check("dfs_select_verify", load().dfs_select_verify(
        ctypes.byref(dims), _ptr(hidden), _ptr(W_vocab), _ptr(W_g), _ptr(A), _ptr(Btab),
        _ptr(last_verified), _ptr(target_logits), int(path_mode), float(temperature),
        int(seed) & (2**64 - 1), _ptr(path), _ptr(out), _ptr(acc), _ptr(ids), _ptr(U), _ptr(S),
        _ptr(score), _ptr(ws), ws.numel(), _stream(stream)))
    res = {"path": path, "out_tokens": out, "accept_len": acc}
    if want_intermediates:
        res.update(cand_ids=ids, cand_U=U, S=S, path_score=score)
    return res


# ---- E4M3 LM head
def dfs_quantize_rows_e4m3(dims: Dims, hidden, stream=None):
    """hidden [B, L, d] bf16 -> (q [B*L, d] uint8 E4M3 bytes, scale [B*L] fp32)."""
    rows = dims.B * dims.L
    q = torch.empty(rows, dims.d, dtype=torch.uint8, device=hidden.device)
    sc = torch.empty(rows, dtype=torch.float32, device=hidden.device)
    _check("dfs_quantize_rows_e4m3", load().dfs_quantize_rows_e4m3(
        ctypes.byref(dims), _ptr(hidden), _ptr(q), _ptr(sc), _stream(stream)))
    return q, sc


def dfs_pack_e4m3_head(Wq, stream=None):
    """Wq [V, d] uint8 E4M3 bytes (row-major, on the device) -> the packed head the E4M3 LM
    head reads (dfs_e4m3_head_bytes(V, d) uint8)."""
    V, d = Wq.shape
    n = load().dfs_e4m3_head_bytes(V, d)
    if n == 0:
        raise DfsError("dfs_e4m3_head_bytes", DFS_ERR_UNSUPPORTED)
    out = torch.empty(n, dtype=torch.uint8, device=Wq.device)
    _check("dfs_pack_e4m3_head", load().dfs_pack_e4m3_head(V, d, _ptr(Wq), _ptr(out),
                                                           _stream(stream)))
    return out


def dfs_next_tokens(out_tokens, accept_len, next_last_verified=None, stream=None):
    """The last token each request emitted (out_tokens [B, L], accept_len [B]) -> [B] int32,
    written into `next_last_verified` when given (e.g. the next cycle's x0 buffer)."""
    B, L = out_tokens.shape
    if next_last_verified is None:
        next_last_verified = torch.empty(B, dtype=torch.int32, device=out_tokens.device)
    _check("dfs_next_tokens", load().dfs_next_tokens(B, L, _ptr(out_tokens), _ptr(accept_len),
                                                     _ptr(next_last_verified), _stream(stream)))
    return next_last_verified


def alloc_conv_workspace(B: int, L: int, d: int, device=None, stream=None) -> torch.Tensor:
    """A zero-initialised workspace for dfs_conv2tap on [B, L, d] inputs."""
    n = load().dfs_conv2tap_workspace_size(B, L, d)
    if n == 0:
        raise DfsError("dfs_conv2tap_workspace_size", DFS_ERR_UNSUPPORTED)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check("dfs_workspace_init", load().dfs_workspace_init(_ptr(ws), n, _stream(stream)))
    return ws


def dfs_conv2tap(x, base, Wc, ws, out=None, stream=None):
    """Two-tap dynamic depthwise convolution: x [B, L, d] bf16, base [2, d] fp32, Wc [d/8, d]
    bf16 -> out [B, L, d] bf16 (written into `out` when given)."""
    B, L, d = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check("dfs_conv2tap", load().dfs_conv2tap(B, L, d, _ptr(x), _ptr(base), _ptr(Wc), _ptr(out),
                                               _ptr(ws), ws.numel(), _stream(stream)))
    return out


def dfs_lmhead_topk_e4m3(dims: Dims, hidden, Wq, w_scale, ws, stream=None):
    P = dims.L - 1
    ids = torch.empty(dims.B, P, K, dtype=torch.int32, device=hidden.device)
    U = torch.empty(dims.B, P, K, dtype=torch.float32, device=hidden.device)
    _check("dfs_lmhead_topk_e4m3", load().dfs_lmhead_topk_e4m3(
        ctypes.byref(dims), _ptr(hidden), _ptr(Wq), _ptr(w_scale), _ptr(ids), _ptr(U), _ptr(ws),
        ws.numel(), _stream(stream)))
    return ids, U


def dfs_select_verify_e4m3(dims: Dims, hidden, Wq, w_scale, W_g, A, Btab, last_verified,
                           target_logits, path_mode: int, temperature: float, seed: int, ws, *,
                           outputs=None, want_intermediates: bool = False, stream=None):
    """The fused step with the E4M3 LM head; as dfs_select_verify."""
    P = dims.L - 1
    dev = hidden.device
    if outputs is None:
        outputs = (torch.empty(dims.B, P, dtype=torch.int32, device=dev),
                   torch.empty(dims.B, dims.L, dtype=torch.int32, device=dev),
                   torch.empty(dims.B, dtype=torch.int32, device=dev))
    path, out, acc = outputs
    ids = U = S = score = None
    if want_intermediates:
        ids = torch.empty(dims.B, P, K, dtype=torch.int32, device=dev)
        U = torch.empty(dims.B, P, K, dtype=torch.float32, device=dev)
        S = torch.empty(dims.B, P, K, K, dtype=torch.float32, device=dev)
        score = torch.empty(dims.B, dtype=torch.float32, device=dev)
    _check("dfs_select_verify_e4m3", load().dfs_select_verify_e4m3(
        ctypes.byref(dims), _ptr(hidden), _ptr(Wq), _ptr(w_scale), _ptr(W_g), _ptr(A),
        _ptr(Btab), _ptr(last_verified), _ptr(target_logits), int(path_mode), float(temperature),
        int(seed) & (2**64 - 1), _ptr(path), _ptr(out), _ptr(acc), _ptr(ids), _ptr(U), _ptr(S),
        _ptr(score), _ptr(ws), ws.numel(), _stream(stream)))
    res = {"path": path, "out_tokens": out, "accept_len": acc}
    if want_intermediates:
        res.update(cand_ids=ids, cand_U=U, S=S, path_score=score)
    return res
