"""fp64 CPU oracle for the draft-block select-and-verify step (DFlash 2).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py --impl reference`` and the
``cpu_baseline`` field) may import this package. The product path (the CUDA
library and its binding) never imports it and shares no code with it.

This module only builds ``oracle.cpp`` with the system C++ compiler and
marshals numpy arrays into it; all arithmetic is in ``oracle.cpp``. Inputs are
numpy arrays: bf16 data is passed as ``uint16`` bit patterns, fp32 as
``float32``. Results are float64 / int32 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, FP32 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.cpp into oracle/_build/liboracle.so (no -ffast-math,
    no FMA contraction, so results match across x86 and Arm hosts)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f64, u64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_uint64
            sig = {
                "orc_abi_version": ([], i32),
                "orc_logits": ([i32, P, P, i64, i64, P, i64, P, i32], i32),
                "orc_topk": ([P, i64, i64, i32, P, P, P], i32),
                "orc_gate": ([i32, P, P, i64, i64, P, i64, P], i32),
                "orc_conv2tap": ([i32, P, P, i32, P, i64, i64, i64, P], i32),
                "orc_pair_scores": ([i32, P, P, i64, i32, i32, P, P, P, ctypes.c_int32, P], i32),
                "orc_path_greedy": ([i32, i32, P, P, P, P, P, P], i32),
                "orc_path_viterbi": ([i32, i32, P, P, P, P, P, P], i32),
                "orc_verify_greedy": ([i32, P, i32, i64, P, P, P], i32),
                "orc_verify_sampling": ([i32, P, i32, i64, P, f64, u64, i64, P, P, P, P], i32),
                "orc_verify_sampling_many": ([i32, P, i32, i64, P, f64, u64, i64, i64, i32, P, P], i32),
                "orc_path_sample": ([i32, i32, P, P, f64, u64, i64, P, P, P, P, P], i32),
                "orc_verify_proposal": ([i32, P, i32, i64, P, P, P, P, i32, f64, u64, i64, P, P,
                                         P, P], i32),
                "orc_sample_verify_many": ([i32, P, i32, i64, P, P, i32, f64, u64, i64, i64, i32,
                                            i32, P, P, P], i32),
                "orc_path_sample_joint": ([i32, i32, P, P, f64, u64, i64, P, P, P, P, P], i32),
                "orc_philox4x64": ([P, P, P], None),
                "orc_redraw_uniforms": ([i32, P, i64, f64, i64, P, P, i32, P, i64, P, P], i32),
                "orc_select_verify": ([i32, i32, P, P, P, P, P, P, P, i64, i32, i64, i64, i64,
                                       i32, i32, f64, u64, P, i64, i32] + [P] * 14, i32),
                "orc_e4m3_decode": ([P, i64, P], None),
                "orc_e4m3_encode": ([P, i64, P], None),
                "orc_quantize_rows_e4m3": ([i32, P, i64, P, i64, P, P], i32),
                "orc_logits_e4m3": ([P, P, P, P, i64, i64, i64, P, i32], i32),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return FP32
    raise TypeError(f"oracle inputs must be uint16 (bf16 bits) or float32, got {a.dtype}")


def _c(a, dtype=None):
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def logits(h, W, rows, nthreads: int | None = None) -> np.ndarray:
    """u[i, v] = sum_k h2[rows[i], k] * W[k, v] in float64; h2 = h viewed as [-1, d]."""
    W = _c(W)
    d, V = W.shape
    h = _c(h).reshape(-1, d)
    if h.dtype != W.dtype:
        raise TypeError("h and W must share a dtype")
    rows = _c(rows, np.int64).reshape(-1)
    u = np.empty((rows.size, V), np.float64)
    _check(_load().orc_logits(_dtype_code(W), _ptr(h), _ptr(W), d, V, _ptr(rows), rows.size,
                              _ptr(u), nthreads or default_threads()), "logits")
    return u


def topk(u, K: int = 16):
    """Top-K by (value desc, id asc) of each row: (ids int32 [n,K], U f64 [n,K], gap f64 [n])."""
    u = _c(u, np.float64)
    n, V = u.shape
    ids = np.empty((n, K), np.int32)
    U = np.empty((n, K), np.float64)
    gap = np.empty(n, np.float64)
    _check(_load().orc_topk(_ptr(u), n, V, K, _ptr(ids), _ptr(U), _ptr(gap)), "topk")
    return ids, U, gap


def gate(h, Wg, rows) -> np.ndarray:
    """g[i, j] = sigmoid(sum_k Wg[j, k] * h2[rows[i], k]) in float64."""
    Wg = _c(Wg)
    r, d = Wg.shape
    h = _c(h).reshape(-1, d)
    rows = _c(rows, np.int64).reshape(-1)
    g = np.empty((rows.size, r), np.float64)
    _check(_load().orc_gate(_dtype_code(Wg), _ptr(h), _ptr(Wg), d, r, _ptr(rows), rows.size,
                            _ptr(g)), "gate")
    return g


def conv2tap(x, base, Wc) -> np.ndarray:
    """Two-tap dynamic depthwise convolution of x [B, L, d] (bf16 bits or fp32) with the base
    kernel base [2, d] (fp32) and the correction map Wc [d/8, d] (bf16 bits or fp32):
    out[b, t] = (base[0] + corr0) * x[b, t] + (base[1] + corr1) * x[b, t-1], x[b, -1] = 0,
    corr = Wc x[b, t] with one value per 16 channels and tap. float64 [B, L, d]."""
    x = _c(x)
    B, L, d = x.shape
    base = _c(base, np.float32).reshape(2, d)
    Wc = _c(Wc).reshape(d // 8, d)
    out = np.empty((B, L, d), np.float64)
    _check(_load().orc_conv2tap(_dtype_code(x), _ptr(x), _ptr(base), _dtype_code(Wc), _ptr(Wc),
                                B, L, d, _ptr(out)), "conv2tap")
    return out


def pair_scores(A, Bt, ids, U, g, x0: int) -> np.ndarray:
    """S[p, a, b] for one request; ids/U [P, K], g [P, r]."""
    A = _c(A)
    Bt = _c(Bt)
    V, r = A.shape
    ids = _c(ids, np.int32)
    P, K = ids.shape
    U = _c(U, np.float64)
    g = _c(g, np.float64)
    assert U.shape == (P, K) and g.shape == (P, r) and Bt.shape == A.shape
    S = np.empty((P, K, K), np.float64)
    _check(_load().orc_pair_scores(_dtype_code(A), _ptr(A), _ptr(Bt), r, P, K, _ptr(ids), _ptr(U),
                                   _ptr(g), int(x0), _ptr(S)), "pair_scores")
    return S


def _path(fn_name, S, ids):
    S = _c(S, np.float64)
    ids = _c(ids, np.int32)
    P, K = ids.shape
    assert S.shape == (P, K, K)
    path = np.empty(P, np.int32)
    pidx = np.empty(P, np.int32)
    score = np.zeros(1, np.float64)
    margin = np.zeros(1, np.float64)
    _check(getattr(_load(), fn_name)(P, K, _ptr(S), _ptr(ids), _ptr(path), _ptr(pidx),
                                     _ptr(score), _ptr(margin)), fn_name)
    return path, pidx, float(score[0]), float(margin[0])


def path_greedy(S, ids):
    """(path tokens [P], candidate indices [P], score, relative margin)."""
    return _path("orc_path_greedy", S, ids)


def path_viterbi(S, ids):
    """(path tokens [P], candidate indices [P], score, relative margin)."""
    return _path("orc_path_viterbi", S, ids)


def verify_greedy(Z, path):
    """Z [L, V] for one request; returns (out [L] int32, accept_len)."""
    Z = _c(Z)
    L, V = Z.shape
    path = _c(path, np.int32)
    out = np.empty(L, np.int32)
    acc = np.zeros(1, np.int32)
    _check(_load().orc_verify_greedy(_dtype_code(Z), _ptr(Z), L, V, _ptr(path), _ptr(out), _ptr(acc)),
           "verify_greedy")
    return out, int(acc[0])


def verify_sampling(Z, path, T: float, seed: int, b: int = 0):
    """Z [L, V] for request index b; returns (out, accept_len, acc_margin, draw_margin)."""
    Z = _c(Z)
    L, V = Z.shape
    path = _c(path, np.int32)
    out = np.empty(L, np.int32)
    acc = np.zeros(1, np.int32)
    am = np.zeros(1, np.float64)
    gm = np.full(1, np.inf, np.float64)
    _check(_load().orc_verify_sampling(_dtype_code(Z), _ptr(Z), L, V, _ptr(path), float(T),
                                       ctypes.c_uint64(seed & (2**64 - 1)), int(b), _ptr(out),
                                       _ptr(acc), _ptr(am), _ptr(gm)), "verify_sampling")
    return out, int(acc[0]), float(am[0]), float(gm[0])


def verify_sampling_many(Z, path, T: float, seed0: int, n: int, b: int = 0,
                         nthreads: int | None = None):
    """Sampling verification for seeds seed0..seed0+n-1: (out [n, L], accept_len [n])."""
    Z = _c(Z)
    L, V = Z.shape
    path = _c(path, np.int32)
    out = np.empty((n, L), np.int32)
    acc = np.empty(n, np.int32)
    _check(_load().orc_verify_sampling_many(_dtype_code(Z), _ptr(Z), L, V, _ptr(path), float(T),
                                            ctypes.c_uint64(seed0), int(n), int(b),
                                            nthreads or default_threads(), _ptr(out), _ptr(acc)),
           "verify_sampling_many")
    return out, acc


def path_sample(S, ids, T: float, seed: int, b: int = 0):
    """Sampled traversal of one request's lattice S [P, K, K], ids [P, K]: (path [P],
    pidx [P], q [P, K], score, margin)."""
    S = _c(S, np.float64)
    P, K, _ = S.shape
    ids = _c(ids, np.int32)
    path = np.empty(P, np.int32)
    pidx = np.empty(P, np.int32)
    q = np.empty((P, K), np.float64)
    sc = np.zeros(1, np.float64)
    mg = np.zeros(1, np.float64)
    _check(_load().orc_path_sample(P, K, _ptr(S), _ptr(ids), float(T),
                                   ctypes.c_uint64(seed & (2**64 - 1)), int(b), _ptr(path),
                                   _ptr(pidx), _ptr(q), _ptr(sc), _ptr(mg)), "path_sample")
    return path, pidx, q, float(sc[0]), float(mg[0])


def path_sample_joint(S, ids, T: float, seed: int, b: int = 0):
    """Joint path draw over one request's lattice S [P, K, K], ids [P, K]: (path [P],
    pidx [P], q [P, K], score, margin)."""
    S = _c(S, np.float64)
    P, K, _ = S.shape
    ids = _c(ids, np.int32)
    path = np.empty(P, np.int32)
    pidx = np.empty(P, np.int32)
    q = np.empty((P, K), np.float64)
    sc = np.zeros(1, np.float64)
    mg = np.zeros(1, np.float64)
    _check(_load().orc_path_sample_joint(P, K, _ptr(S), _ptr(ids), float(T),
                                         ctypes.c_uint64(seed & (2**64 - 1)), int(b), _ptr(path),
                                         _ptr(pidx), _ptr(q), _ptr(sc), _ptr(mg)),
           "path_sample_joint")
    return path, pidx, q, float(sc[0]), float(mg[0])


def verify_proposal(Z, path, cand, q, pidx, T: float, seed: int, b: int = 0):
    """Z [L, V]; the proposal's candidates cand [P, K], distributions q [P, K] and drawn
    indices pidx [P]: (out, accept_len, acc_margin, draw_margin)."""
    Z = _c(Z)
    L, V = Z.shape
    cand = _c(cand, np.int32)
    K = cand.shape[1]
    q = _c(q, np.float64)
    out = np.empty(L, np.int32)
    acc = np.zeros(1, np.int32)
    am = np.zeros(1, np.float64)
    gm = np.full(1, np.inf, np.float64)
    _check(_load().orc_verify_proposal(_dtype_code(Z), _ptr(Z), L, V, _ptr(_c(path, np.int32)),
                                       _ptr(cand), _ptr(q), _ptr(_c(pidx, np.int32)), K, float(T),
                                       ctypes.c_uint64(seed & (2**64 - 1)), int(b), _ptr(out),
                                       _ptr(acc), _ptr(am), _ptr(gm)), "verify_proposal")
    return out, int(acc[0]), float(am[0]), float(gm[0])


def sample_verify_many(Z, S, ids, T: float, seed0: int, n: int, b: int = 0,
                       nthreads: int | None = None, joint: bool = False):
    """Sampled traversal (joint: the joint path draw) + its verification for seeds
    seed0..seed0+n-1 on a fixed lattice: (paths [n, P], out [n, L], accept_len [n])."""
    Z = _c(Z)
    L, V = Z.shape
    S = _c(S, np.float64)
    ids = _c(ids, np.int32)
    K = ids.shape[1]
    paths = np.empty((n, L - 1), np.int32)
    out = np.empty((n, L), np.int32)
    acc = np.empty(n, np.int32)
    _check(_load().orc_sample_verify_many(_dtype_code(Z), _ptr(Z), L, V, _ptr(S), _ptr(ids), K,
                                          float(T), ctypes.c_uint64(seed0), int(n), int(b),
                                          nthreads or default_threads(), int(bool(joint)),
                                          _ptr(paths), _ptr(out), _ptr(acc)),
           "sample_verify_many")
    return paths, out, acc


def redraw_uniforms(z, T: float, u, excl: int = -1, cand=None, q=None):
    """The verification's redraw of one target row z [V] for the given uniforms u [n]:
    without cand, a draw from softmax(z/T) with token excl removed; with cand [K] and q [K],
    a draw from the residual max(0, p - q). Returns (tokens int64 [n], margins f64 [n])."""
    z = _c(z).reshape(-1)
    u = _c(u, np.float64).reshape(-1)
    out = np.empty(u.size, np.int64)
    mg = np.empty(u.size, np.float64)
    K = 0 if cand is None else len(cand)
    cand = _c(cand if cand is not None else np.zeros(1), np.int32)
    q = _c(q if q is not None else np.zeros(1), np.float64)
    _check(_load().orc_redraw_uniforms(_dtype_code(z), _ptr(z), z.size, float(T), int(excl),
                                       _ptr(cand), _ptr(q), K, _ptr(u), u.size, _ptr(out),
                                       _ptr(mg)), "redraw_uniforms")
    return out, mg


def philox4x64(ctr, key) -> np.ndarray:
    """One Philox4x64-10 block: counter (4 x uint64), key (2 x uint64) -> 4 x uint64."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    o = np.empty(4, np.uint64)
    _load().orc_philox4x64(_ptr(c), _ptr(k), _ptr(o))
    return o


def e4m3_decode(b) -> np.ndarray:
    """E4M3 bytes -> float64 (OCP OFP8)."""
    b = _c(b, np.uint8).reshape(-1)
    out = np.empty(b.size, np.float64)
    _load().orc_e4m3_decode(_ptr(b), b.size, _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """float64 values (|x| <= 448) -> E4M3 bytes, round to nearest even."""
    x = _c(x, np.float64).reshape(-1)
    out = np.empty(x.size, np.uint8)
    _load().orc_e4m3_encode(_ptr(x), x.size, _ptr(out))
    return out


def quantize_rows_e4m3(h, rows):
    """h viewed as [-1, d]; (q [n, d] uint8, scale [n] float64)."""
    h = _c(h)
    d = h.shape[-1]
    h2 = h.reshape(-1, d)
    rows = _c(rows, np.int64).reshape(-1)
    q = np.empty((rows.size, d), np.uint8)
    sc = np.empty(rows.size, np.float64)
    _check(_load().orc_quantize_rows_e4m3(_dtype_code(h2), _ptr(h2), d, _ptr(rows), rows.size,
                                          _ptr(q), _ptr(sc)), "quantize_rows_e4m3")
    return q, sc


def logits_e4m3(q, h_scale, Wq, w_scale, nthreads: int | None = None) -> np.ndarray:
    """u [n, V] from quantised rows q [n, d] (scales h_scale [n]) and the E4M3 LM head
    Wq [V, d] (scales w_scale [V])."""
    q = _c(q, np.uint8)
    n, d = q.shape
    Wq = _c(Wq, np.uint8)
    V = Wq.shape[0]
    u = np.empty((n, V), np.float64)
    _check(_load().orc_logits_e4m3(_ptr(q), _ptr(_c(h_scale, np.float64)), _ptr(Wq),
                                   _ptr(_c(w_scale, np.float32)), d, V, n, _ptr(u),
                                   nthreads or default_threads()), "logits_e4m3")
    return u


def select_verify(h, W, Wg, A, Bt, x0, Z, *, K: int = 16, path_mode: int = 0,
                  temperature: float = 0.0, seed: int = 0, reqs=None,
                  nthreads: int | None = None, Wq=None, w_scale=None) -> dict:
    """The whole step for the listed requests (default: all).

    h [B, L, d], W [d, V], Wg [r, d], A/Bt [V, r] share one dtype (uint16 = bf16 bits,
    or float32); Z [B, L, V] may be either; x0 [B] int. Returns a dict of numpy arrays
    indexed by list position."""
    h = _c(h)
    B, L, d = h.shape
    W = _c(W)
    V = W.shape[1]
    Wg = _c(Wg)
    r = Wg.shape[0]
    A = _c(A)
    Bt = _c(Bt)
    Z = _c(Z)
    x0 = _c(x0, np.int32)
    dt = _dtype_code(W)
    if not (h.dtype == W.dtype == Wg.dtype == A.dtype == Bt.dtype):
        raise TypeError("h, W, Wg, A and Bt must share a dtype")
    reqs = np.arange(B, dtype=np.int64) if reqs is None else _c(reqs, np.int64).reshape(-1)
    n = reqs.size
    P = L - 1
    res = {
        "cand_ids": np.empty((n, P, K), np.int32),
        "cand_U": np.empty((n, P, K), np.float64),
        "gate": np.empty((n, P, r), np.float64),
        "S": np.empty((n, P, K, K), np.float64),
        "path": np.empty((n, P), np.int32),
        "path_score": np.empty(n, np.float64),
        "out_tokens": np.empty((n, L), np.int32),
        "accept_len": np.empty(n, np.int32),
        "topk_gap": np.empty((n, P), np.float64),
        "path_margin": np.empty(n, np.float64),
        "acc_margin": np.empty(n, np.float64),
        "draw_margin": np.empty(n, np.float64),
    }
    order = ["cand_ids", "cand_U", "gate", "S", "path", "path_score", "out_tokens", "accept_len",
             "topk_gap", "path_margin", "acc_margin", "draw_margin"]
    if Wq is not None:
        Wq = _c(Wq, np.uint8)
        w_scale = _c(w_scale, np.float32)
    rc = _load().orc_select_verify(
        dt, _dtype_code(Z), _ptr(h), _ptr(W), _ptr(Wg), _ptr(A), _ptr(Bt), _ptr(x0), _ptr(Z),
        B, L, V, d, r, K, int(path_mode), float(temperature), ctypes.c_uint64(seed & (2**64 - 1)),
        _ptr(reqs), n, nthreads or default_threads(), *[_ptr(res[k]) for k in order],
        None if Wq is None else _ptr(Wq), None if w_scale is None else _ptr(w_scale))
    _check(rc, "select_verify")
    res["reqs"] = reqs
    return res
