"""CPU oracle for the speculative-decoding verify step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never loads it and shares
no code with it.  The arithmetic lives in ``oracle.c`` (plain C, double
precision, naive loops); this module only marshals numpy arrays into it, and
``toy_model.py`` adds the greedy / speculative decode loops of a toy target.

What each function restates is cited in ``oracle.c``: "Efficient LLM
Challenge Results" (AdaptFM @ ICML 2026), section 3 "Speculative decoding did
the heavy lifting" and section 5 "Quantization was common, but not the
deciding lever".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd[:5] + ["-fopenmp"] + cmd[5:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(cmd, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the argument types of the C entry points on a loaded library."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_dequant_w4.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_w4a16_gemm.argtypes = [P, P, P, P, I, I, I, I, P, P]
    lib.oracle_matmul_dequantized.argtypes = [P, P, I, I, I, P]
    lib.oracle_w4a16_gemm_sampled.argtypes = [P, P, P, P, I, I, I, P, P, I, P]
    lib.oracle_lmhead_logits.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_lmhead_argmax_rows.argtypes = [P, P, P, I, I, P, I, P, P, P]
    lib.oracle_argmax_f64.argtypes = [P, I, I, P]
    lib.oracle_argmax_f32.argtypes = [P, I, I, P]
    lib.oracle_spec_accept.argtypes = [P, P, I, I, P, P]
    lib.oracle_ngram_draft.argtypes = [P, P, I, I, I, I, I, P, P]
    lib.oracle_gdn_recurrence.argtypes = [P, P, P, P, P, P, I, I, I, P, P]
    lib.oracle_num_threads.restype = I
    lib.oracle_set_num_threads.argtypes = [I]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _use_library(path: str) -> None:
    """Route every function of this module through another build of oracle.c
    (the pin tests run this way against copies with a planted mistake)."""
    global _lib
    with _lock:
        _lib = _bind(ctypes.CDLL(path))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _half_bits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError("expected float16 (or its uint16 bit pattern), got %s" % a.dtype)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits) & 0xFFFF)


def dequant_w4(q, s, zeros=None, group=128):
    """w[n][k] = s[k/G][n] * (q[n][k] - z), z = 8 unless a [K/G][N] zero table is given."""
    q = _c(q, np.uint8)
    N, K = q.shape
    s = _half_bits(s)
    assert s.shape == (K // group, N)
    z = None if zeros is None else _c(zeros, np.uint8)
    w = np.empty((N, K), np.float64)
    _load().oracle_dequant_w4(_ptr(q), _ptr(s), _ptr(z), N, K, group, _ptr(w))
    return w


def w4a16_gemm(A, q, s, zeros=None, group=128):
    """C = A @ deq(q, s)^T in double; A fp16 [M][K], q uint8 codes [N][K], s fp16 [K/G][N]."""
    A = _half_bits(A)
    q = _c(q, np.uint8)
    M, K = A.shape
    N = q.shape[0]
    assert q.shape == (N, K) and K % group == 0
    s = _half_bits(s)
    assert s.shape == (K // group, N)
    z = None if zeros is None else _c(zeros, np.uint8)
    w = np.empty((N, K), np.float64)
    C = np.empty((M, N), np.float64)
    _load().oracle_w4a16_gemm(_ptr(A), _ptr(q), _ptr(s), _ptr(z), group, M, N, K, _ptr(w), _ptr(C))
    return C


def matmul_dequantized(A, w):
    """C = A @ w^T in double for fp16 A [M][K] and a dequantized double w [N][K]."""
    A = _half_bits(A)
    w = _c(w, np.float64)
    M, K = A.shape
    N = w.shape[0]
    assert w.shape == (N, K)
    C = np.empty((M, N), np.float64)
    _load().oracle_matmul_dequantized(_ptr(A), _ptr(w), M, N, K, _ptr(C))
    return C


def w4a16_gemm_sampled(A, q, s, rows, cols, zeros=None, group=128):
    """C[rows[i]][cols[i]] for each i, from the same definition (no full product)."""
    A = _half_bits(A)
    q = _c(q, np.uint8)
    N, K = q.shape
    s = _half_bits(s)
    rows = _c(rows, np.int32)
    cols = _c(cols, np.int32)
    z = None if zeros is None else _c(zeros, np.uint8)
    out = np.empty(rows.shape[0], np.float64)
    _load().oracle_w4a16_gemm_sampled(_ptr(A), _ptr(q), _ptr(s), _ptr(z), group, N, K,
                                      _ptr(rows), _ptr(cols), rows.shape[0], _ptr(out))
    return out


def lmhead_logits(X, W, s):
    """L[r][v] = s[v] * sum_k X[r][k] W[v][k] in double; X fp16 [M][K], W int8 [V][K], s fp16 [V]."""
    X = _half_bits(X)
    W = _c(W, np.int8)
    M, K = X.shape
    V = W.shape[0]
    assert W.shape == (V, K)
    s = _half_bits(s)
    assert s.shape == (V,)
    L = np.empty((M, V), np.float64)
    _load().oracle_lmhead_logits(_ptr(X), _ptr(W), _ptr(s), M, K, V, _ptr(L))
    return L


def lmhead_argmax_rows(X, W, s, rows):
    """(token, best logit, second-best logit) for the listed rows of X, in double."""
    X = _half_bits(X)
    W = _c(W, np.int8)
    K = X.shape[1]
    V = W.shape[0]
    s = _half_bits(s)
    rows = _c(rows, np.int32)
    n = rows.shape[0]
    tok = np.empty(n, np.int32)
    best = np.empty(n, np.float64)
    second = np.empty(n, np.float64)
    _load().oracle_lmhead_argmax_rows(_ptr(X), _ptr(W), _ptr(s), K, V, _ptr(rows), n,
                                      _ptr(tok), _ptr(best), _ptr(second))
    return tok, best, second


def argmax(L):
    """Row-wise greedy token: lowest index among maxima, NaN counted as -inf."""
    L = np.ascontiguousarray(L)
    if L.ndim == 1:
        return int(argmax(L[None, :])[0])
    M, V = L.shape
    out = np.empty(M, np.int32)
    if L.dtype == np.float32:
        _load().oracle_argmax_f32(_ptr(L), M, V, _ptr(out))
    else:
        L = _c(L, np.float64)
        _load().oracle_argmax_f64(_ptr(L), M, V, _ptr(out))
    return out


def spec_accept(target, draft):
    """Longest-prefix greedy acceptance.

    target int32 [B][K+1], draft int32 [B][K] (negative = padding sentinel).
    Returns (n [B], tokens [B][K+1]) where tokens[b][:n+1] are the emitted
    tokens and the rest are -1.  1-D inputs give (int n, tokens [K+1]).
    """
    t = _c(target, np.int32)
    d = _c(draft, np.int32)
    if t.ndim == 1:
        n, tok = spec_accept(t[None, :], d.reshape(1, -1))
        return int(n[0]), tok[0]
    B, K1 = t.shape
    K = K1 - 1
    d = d.reshape(B, K)
    n = np.empty(B, np.int32)
    tok = np.empty((B, K + 1), np.int32)
    _load().oracle_spec_accept(_ptr(t), _ptr(d), B, K, _ptr(n), _ptr(tok))
    return n, tok


def ngram_draft(context, lengths, n_min, n_max, K):
    """Prompt-lookup drafts for each row of context int32 [B][ld] (row b holds
    lengths[b] tokens): (drafts int32 [B][K] with -1 padding, match length [B])."""
    c = _c(context, np.int32)
    if c.ndim == 1:
        d, m = ngram_draft(c[None, :], [c.shape[0]], n_min, n_max, K)
        return d[0], int(m[0])
    B, ld = c.shape
    ln = _c(lengths, np.int32).reshape(B)
    assert np.all((ln >= 0) & (ln <= ld)) and 1 <= n_min <= n_max and K >= 0
    d = np.empty((B, K), np.int32)
    m = np.empty(B, np.int32)
    _load().oracle_ngram_draft(_ptr(c), _ptr(ln), B, ld, int(n_min), int(n_max), int(K), _ptr(d), _ptr(m))
    return d, m


def gdn_recurrence(S0, q, k, v, alpha, beta):
    """Gated delta recurrence per head, in double:
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t.
    S0 [H][dv][dk]; q, k [T][H][dk]; v [T][H][dv]; alpha, beta [T][H] (any float dtype,
    converted exactly to double).  Returns (o [T][H][dv], S_T [H][dv][dk])."""
    S0 = _c(S0, np.float64)
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    alpha = _c(alpha, np.float64)
    beta = _c(beta, np.float64)
    H, dv, dk = S0.shape
    T = q.shape[0]
    assert q.shape == (T, H, dk) and k.shape == (T, H, dk) and v.shape == (T, H, dv)
    assert alpha.shape == (T, H) and beta.shape == (T, H)
    o = np.empty((T, H, dv), np.float64)
    S = np.empty((H, dv, dk), np.float64)
    lib = _load()
    for h in range(H):
        qh, kh, vh = _c(q[:, h], np.float64), _c(k[:, h], np.float64), _c(v[:, h], np.float64)
        ah, bh = _c(alpha[:, h], np.float64), _c(beta[:, h], np.float64)
        oh = np.empty((T, dv), np.float64)
        Sh = np.empty((dv, dk), np.float64)
        lib.oracle_gdn_recurrence(_ptr(_c(S0[h], np.float64)), _ptr(qh), _ptr(kh), _ptr(vh), _ptr(ah), _ptr(bh),
                                  T, dk, dv, _ptr(oh), _ptr(Sh))
        o[:, h] = oh
        S[h] = Sh
    return o, S
