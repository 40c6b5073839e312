"""ctypes marshalling for the C oracle (``wide_oracle.c``).

Test infrastructure only: the product path never reaches this module.
Arrays are numpy; bf16 tensors travel as their raw ``uint16`` bit patterns,
masks as ``uint8``; floating-point outputs come back as ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wide_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "libwide_oracle.so")
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over tokens); returns the .so path."""
    with _lock:
        stale = (not os.path.exists(_LIB)
                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if force or stale:
            os.makedirs(_BUILD_DIR, exist_ok=True)
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                   _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_version.restype = i
        lib.oracle_reorder.argtypes = [p, i, i, p, p]
        lib.oracle_reorder.restype = None
        for name in ("oracle_proj_mn", "oracle_proj_k"):
            getattr(lib, name).argtypes = [p, p, p, i, i, i, i, p, i, p]
            getattr(lib, name).restype = None
        lib.oracle_gate_up.argtypes = [p, p, p, p, i, i, i, i, p, i, p]
        lib.oracle_gate_up.restype = None
        lib.oracle_ffn.argtypes = [p, p, p, p, p, i, i, i, i, p, i, p, p]
        lib.oracle_ffn.restype = None
        lib.oracle_router.argtypes = [p, p, p, i, i, i, i, p, p]
        lib.oracle_router.restype = None
        lib.oracle_attn_decode.argtypes = [p, p, p, p, p, i, i, i, i, i, p]
        lib.oracle_attn_decode.restype = None
        lib.oracle_attn_prefill.argtypes = [p, p, p, p, i, i, i, i, i, i, p, i, p]
        lib.oracle_attn_prefill.restype = None
        _lib = lib
    return _lib


def threads() -> int:
    """Number of OpenMP threads the oracle will use (OMP_NUM_THREADS or cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env:
        return int(env)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _rows(rows, T):
    if rows is None:
        return None, T
    r = _c(rows, np.int32)
    if r.ndim != 1 or (r.size and (r.min() < 0 or r.max() >= T)):
        raise ValueError("rows must be a 1-D list of token indices in [0, T)")
    return r, int(r.size)


def reorder(mask: np.ndarray):
    """Eq. 7 SortDesc per routing column -> (perm [n_groups, T], counts [n_groups])."""
    m = _c(mask, np.uint8)
    T, n_groups = m.shape
    perm = np.empty((n_groups, T), np.int32)
    counts = np.empty((n_groups,), np.int32)
    _load().oracle_reorder(_ptr(m), T, n_groups, _ptr(perm), _ptr(counts))
    return perm, counts


def proj_mn(X, W, mask, G, rows=None):
    """Y[t,n] = M[t,n/G] * sum_k X[t,k] W[n,k]  (X, W as bf16 bits)."""
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    m = _c(mask, np.uint8)
    T, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K and N % G == 0 and m.shape == (T, N // G)
    r, R = _rows(rows, T)
    Y = np.empty((R, N), np.float64)
    _load().oracle_proj_mn(_ptr(X), _ptr(W), _ptr(m), T, K, N, G,
                           None if r is None else _ptr(r), R, _ptr(Y))
    return Y


def gate_up(X, Wg, Wu, mask, G, rows=None):
    """H[t,f] = M[t,f/G] * silu(X Wg^T)[t,f] * (X Wu^T)[t,f]  (bf16 bits in)."""
    X = _c(X, np.uint16)
    Wg = _c(Wg, np.uint16)
    Wu = _c(Wu, np.uint16)
    m = _c(mask, np.uint8)
    T, D = X.shape
    F = Wg.shape[0]
    assert Wg.shape == (F, D) and Wu.shape == (F, D)
    assert F % G == 0 and m.shape == (T, F // G)
    r, R = _rows(rows, T)
    H = np.empty((R, F), np.float64)
    _load().oracle_gate_up(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(m), T, D, F, G,
                           None if r is None else _ptr(r), R, _ptr(H))
    return H


def proj_k(A, W, mask, G, rows=None):
    """Y[t,n] = sum_g M[t,g] sum_{k in K_g} A[t,k] W[n,k]  (Eq. 21)."""
    A = _c(A, np.uint16)
    W = _c(W, np.uint16)
    m = _c(mask, np.uint8)
    T, K = A.shape
    N = W.shape[0]
    assert W.shape[1] == K and K % G == 0 and m.shape == (T, K // G)
    r, R = _rows(rows, T)
    Y = np.empty((R, N), np.float64)
    _load().oracle_proj_k(_ptr(A), _ptr(W), _ptr(m), T, K, N, G,
                          None if r is None else _ptr(r), R, _ptr(Y))
    return Y


def ffn(X, Wg, Wu, Wd, mask, G, rows=None):
    """Whole masked FFN of Eq. 3, intermediate kept in double."""
    X = _c(X, np.uint16)
    Wg = _c(Wg, np.uint16)
    Wu = _c(Wu, np.uint16)
    Wd = _c(Wd, np.uint16)
    m = _c(mask, np.uint8)
    T, D = X.shape
    F = Wg.shape[0]
    assert Wg.shape == (F, D) and Wu.shape == (F, D) and Wd.shape == (D, F)
    assert F % G == 0 and m.shape == (T, F // G)
    r, R = _rows(rows, T)
    Y = np.empty((R, D), np.float64)
    scratch = np.empty((R, F), np.float64)
    _load().oracle_ffn(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(m),
                       T, D, F, G, None if r is None else _ptr(r), R,
                       _ptr(Y), _ptr(scratch))
    return Y


def router(X, W1, W2):
    """Eq. 4-5: logits R [T, 2*n_groups] (column 2g+c) and mask [T, n_groups].

    X bf16 [T, D], W1 bf16 [r, D], W2 bf16 [2*n_groups, r] (as bit patterns).
    mask[t,g] = R[t,g,0] >= R[t,g,1] with the logits rounded to float."""
    X = _c(X, np.uint16)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    T, D = X.shape
    r = W1.shape[0]
    assert W1.shape == (r, D) and W2.shape[1] == r and W2.shape[0] % 2 == 0 and r <= 1024
    ng = W2.shape[0] // 2
    logits = np.empty((T, 2 * ng), np.float64)
    mask = np.empty((T, ng), np.uint8)
    _load().oracle_router(_ptr(X), _ptr(W1), _ptr(W2), T, D, r, ng, _ptr(logits), _ptr(mask))
    return logits, mask


def attn_decode(Q, K, V, lens, mask):
    """Routed decode attention: O [B, Hq, d] (double).

    Q bf16 [B, Hq, d]; K, V bf16 [B, Hk, L_max, d]; lens int32 [B];
    mask uint8 [B, Hk] (group g = KV head g and its Hq/Hk query heads)."""
    Q = _c(Q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    lens = _c(lens, np.int32)
    m = _c(mask, np.uint8)
    B, Hq, d = Q.shape
    _, Hk, L_max, d2 = K.shape
    assert K.shape == V.shape and K.shape[0] == B and d2 == d and Hq % Hk == 0
    assert lens.shape == (B,) and m.shape == (B, Hk) and (lens <= L_max).all()
    O = np.empty((B, Hq, d), np.float64)
    _load().oracle_attn_decode(_ptr(Q), _ptr(K), _ptr(V), _ptr(lens), _ptr(m), B, Hq, Hk, d,
                               L_max, _ptr(O))
    return O


def attn_prefill(Q, K, V, mask, causal=True, rows=None):
    """Routed prefill attention: O [B, T, Hq, d] (double), or [B, len(rows),
    Hq, d] for a list of token positions `rows` (every sequence, all heads).

    Q bf16 [B, T, Hq, d]; K, V bf16 [B, Hk, T, d]; mask uint8 [B, T, Hk]."""
    Q = _c(Q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    m = _c(mask, np.uint8)
    B, T, Hq, d = Q.shape
    Hk = K.shape[1]
    assert K.shape == (B, Hk, T, d) and V.shape == K.shape and Hq % Hk == 0 and m.shape == (B, T, Hk)
    r, R = _rows(rows, T)
    O = np.empty((B, R, Hq, d), np.float64)
    _load().oracle_attn_prefill(_ptr(Q), _ptr(K), _ptr(V), _ptr(m), B, T, Hq, Hk, d,
                                1 if causal else 0, None if r is None else _ptr(r), R, _ptr(O))
    return O
