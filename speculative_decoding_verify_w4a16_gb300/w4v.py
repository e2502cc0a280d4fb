"""Thin ctypes binding of libw4v (include/w4v.h): argument marshalling only.

Every step of the verify path runs in the library's CUDA kernels; this
module passes device pointers from torch tensors, the current stream, and
turns status codes into exceptions.  There is no fallback: if the library is
missing or the GPU is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libw4v.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "w4v.h")

OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT = range(8)
GROUP = 128

_lock = threading.Lock()
_lib = None


class Problem(ctypes.Structure):
    """w4a16_problem (include/w4v.h)."""
    _fields_ = [("A", ctypes.c_void_p), ("Bq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("C", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int)]


class GroupedHandle(ctypes.Structure):
    """w4a16_grouped_t (include/w4v.h): filled by w4a16_grouped_plan."""
    _fields_ = [("plan", ctypes.c_void_p), ("units", ctypes.c_longlong), ("n_problems", ctypes.c_int),
                ("M", ctypes.c_int), ("group", ctypes.c_int), ("has_zeros", ctypes.c_int), ("tiles", ctypes.c_int),
                ("check", ctypes.c_uint)]


class W4VError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (w4v status %d)" % (where, status_string(code), code))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libw4v.so (built by ``_build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError("libw4v.so not built: run speculative_decoding_verify_w4a16_gb300._build.build()")
            lib = ctypes.CDLL(path)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.w4v_status_string.argtypes = [I]
            lib.w4v_status_string.restype = ctypes.c_char_p
            lib.w4v_init.restype = I
            lib.w4v_get_status.argtypes = [P]
            lib.w4v_get_status.restype = I
            lib.w4v_packed_bytes.argtypes = [I, I]
            lib.w4v_packed_bytes.restype = S
            lib.w4v_pack_int4.argtypes = [P, I, I, P]
            lib.w4v_pack_int4.restype = I
            lib.w4v_unpack_int4.argtypes = [P, I, I, P]
            lib.w4v_unpack_int4.restype = I
            lib.w4a16_workspace_bytes.argtypes = [I, I, I]
            lib.w4a16_workspace_bytes.restype = S
            lib.w4a16_gemm.argtypes = [P, P, P, P, I, P, I, I, I, P, S, P]
            lib.w4a16_gemm.restype = I
            lib.w4a16_gemm_ex.argtypes = [P, P, P, P, I, P, I, I, I, P, S, ctypes.c_uint, P]
            lib.w4a16_gemm_ex.restype = I
            lib.w4a16_grouped_plan_bytes.argtypes = [I]
            lib.w4a16_grouped_plan_bytes.restype = S
            lib.w4a16_grouped_plan.argtypes = [P, I, I, I, P, S, P, P]
            lib.w4a16_grouped_plan.restype = I
            lib.w4a16_grouped_workspace_bytes.argtypes = [P]
            lib.w4a16_grouped_workspace_bytes.restype = S
            lib.w4a16_gemm_grouped.argtypes = [P, P, S, ctypes.c_uint, P]
            lib.w4a16_gemm_grouped.restype = I
            lib.w8_lmhead_argmax_workspace_bytes.argtypes = [I, I]
            lib.w8_lmhead_argmax_workspace_bytes.restype = S
            lib.w8_lmhead_argmax.argtypes = [P, P, P, I, I, I, P, P, P, P, S, P]
            lib.w8_lmhead_argmax.restype = I
            lib.w8_lmhead_argmax_ex.argtypes = [P, P, P, I, I, I, P, P, P, P, S, ctypes.c_uint, P]
            lib.w8_lmhead_argmax_ex.restype = I
            lib.w8_lmhead_argmax_accept_ex.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, S, ctypes.c_uint, P]
            lib.w8_lmhead_argmax_accept_ex.restype = I
            lib.spec_accept.argtypes = [P, P, I, I, P, P, P]
            lib.spec_accept.restype = I
            lib.w8_lmhead_argmax_accept.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, S, P]
            lib.w8_lmhead_argmax_accept.restype = I
            lib.ngram_draft_workspace_bytes.argtypes = [I]
            lib.ngram_draft_workspace_bytes.restype = S
            lib.ngram_draft.argtypes = [P, P, I, I, I, I, I, P, P, P, S, P]
            lib.ngram_draft.restype = I
            lib.gdn_verify.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P]
            lib.gdn_verify.restype = I
            lib.gdn_commit.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P]
            lib.gdn_commit.restype = I
            lib.gdn_step.argtypes = [P, P, P, P, P, P, I, P, P, P, P, P, I, I, I, I, I, P, P]
            lib.gdn_step.restype = I
            _lib = lib
    return _lib


def header_functions(path: str = HEADER):
    """Names of the functions declared in include/w4v.h."""
    with open(path) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text)) -
                  {"if", "defined", "sizeof"})


def status_string(code: int) -> str:
    try:
        return load().w4v_status_string(int(code)).decode()
    except Exception:
        return "status %d" % code


def _check(code: int, where: str) -> None:
    if code != OK:
        raise W4VError(code, where)


def _stream(stream=None) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else s


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def init() -> None:
    _check(load().w4v_init(), "w4v_init")


def get_status(stream=None) -> int:
    return load().w4v_get_status(_stream(stream))


# ------------------------------------------------------------------ packing --
def packed_bytes(N: int, K: int) -> int:
    return load().w4v_packed_bytes(N, K)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Logical codes uint8 [N][K] (0..15) -> the library's packed tile layout (host)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    nbytes = packed_bytes(N, K)
    if nbytes == 0:
        raise W4VError(ERR_SHAPE, "w4v_pack_int4")
    out = np.empty(nbytes, np.uint8)
    _check(load().w4v_pack_int4(q.ctypes.data, N, K, out.ctypes.data), "w4v_pack_int4")
    return out


def unpack_int4(packed: np.ndarray, N: int, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    q = np.empty((N, K), np.uint8)
    _check(load().w4v_unpack_int4(packed.ctypes.data, N, K, q.ctypes.data), "w4v_unpack_int4")
    return q


# --------------------------------------------------------------- workspaces --
def w4a16_workspace_bytes(M: int, N: int, K: int) -> int:
    return load().w4a16_workspace_bytes(M, N, K)


def w8_lmhead_argmax_workspace_bytes(M: int, V: int) -> int:
    return load().w8_lmhead_argmax_workspace_bytes(M, V)


def workspace(nbytes: int, device="cuda"):
    """A zero-filled device workspace (the library leaves it zeroed after each call)."""
    import torch
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ compute --
STATIC_WEIGHTS = 1
BATCH_INVARIANT = 2


def w4a16_gemm(A, Bq, scales, N: int, zeros=None, out=None, ws=None, stream=None, static_weights=False,
               group: int = GROUP, batch_invariant=False):
    """C = A @ deq(Bq, scales, zeros)^T on the GPU.  A fp16 [M][K] cuda, Bq packed uint8 cuda,
    scales fp16 [K/group][N] (group 128 or 32).
    static_weights: the caller promises no GPU work still in flight writes Bq, scales or zeros
    (w4a16_gemm_ex with W4V_STATIC_WEIGHTS).
    batch_invariant: for M > 32, 32-row blocks through the verify-sized kernel
    (W4V_BATCH_INVARIANT): each row equals the row computed alone."""
    import torch
    M, K = A.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    if ws is None:
        ws = workspace(w4a16_workspace_bytes(M, N, K), A.device)
    flags = (STATIC_WEIGHTS if static_weights else 0) | (BATCH_INVARIANT if batch_invariant else 0)
    code = load().w4a16_gemm_ex(_ptr(A), _ptr(Bq), _ptr(scales), _ptr(zeros), int(group), _ptr(out), M, N, K,
                                _ptr(ws), ws.numel(), flags, _stream(stream))
    _check(code, "w4a16_gemm")
    return out


class GroupedGemm:
    """Several independent W4A16 products in one launch (w4a16_grouped_plan +
    w4a16_gemm_grouped).  `problems` is a list of (A, Bq, scales, zeros, C)
    device tensors (zeros None or a uint8 table for every problem), all with
    the same number of rows M; the plan keeps them alive and refers to their
    addresses, so call it again with the same tensors (refill them in place)."""

    def __init__(self, problems, group: int = GROUP, stream=None):
        import torch
        lib = load()
        self.problems = list(problems)
        n = len(self.problems)
        M = self.problems[0][0].shape[0]
        dev = self.problems[0][0].device
        arr = (Problem * n)()
        for i, (A, Bq, sc, z, C) in enumerate(self.problems):
            arr[i] = Problem(_ptr(A), _ptr(Bq), _ptr(sc), _ptr(z), _ptr(C), int(C.shape[1]), int(A.shape[1]))
        nbytes = lib.w4a16_grouped_plan_bytes(n)
        # torch's allocations start on 512-byte boundaries (the plan needs 64)
        self.plan = torch.empty(max(int(nbytes), 64), dtype=torch.uint8, device=dev)
        self.handle = GroupedHandle()
        code = lib.w4a16_grouped_plan(arr, n, int(M), int(group), _ptr(self.plan), self.plan.numel(),
                                      ctypes.byref(self.handle), _stream(stream))
        _check(code, "w4a16_grouped_plan")
        self.ws = workspace(lib.w4a16_grouped_workspace_bytes(ctypes.byref(self.handle)), dev)

    def __call__(self, stream=None, static_weights: bool = False, ws=None):
        ws = self.ws if ws is None else ws
        code = load().w4a16_gemm_grouped(ctypes.byref(self.handle), _ptr(ws), ws.numel(),
                                         STATIC_WEIGHTS if static_weights else 0, _stream(stream))
        _check(code, "w4a16_gemm_grouped")
        return [p[4] for p in self.problems]


def w8_lmhead_argmax(X, W, scale, out=None, maxlogit=None, logits=None, ws=None, stream=None,
                     batch_invariant=False):
    """Greedy token per row of X through the int8 lm_head; returns the int32 [M] token tensor.
    batch_invariant: for M > 32, blocks of 32 rows (W4V_BATCH_INVARIANT): each row's
    logits and token equal those of the row computed alone."""
    import torch
    M, K = X.shape
    V = W.shape[0]
    if out is None:
        out = torch.empty(M, dtype=torch.int32, device=X.device)
    if ws is None:
        ws = workspace(w8_lmhead_argmax_workspace_bytes(M, V), X.device)
    code = load().w8_lmhead_argmax_ex(_ptr(X), _ptr(W), _ptr(scale), M, K, V, _ptr(out), _ptr(maxlogit),
                                      _ptr(logits), _ptr(ws), ws.numel(), BATCH_INVARIANT if batch_invariant else 0,
                                      _stream(stream))
    _check(code, "w8_lmhead_argmax")
    return out


def spec_accept(target, draft, n_out=None, tok_out=None, stream=None):
    """(n [B], tokens [B][K+1]) for int32 target [B][K+1] and drafts [B][K] on the GPU."""
    import torch
    B, K1 = target.shape
    K = K1 - 1
    if n_out is None:
        n_out = torch.empty(B, dtype=torch.int32, device=target.device)
    if tok_out is None:
        tok_out = torch.empty((B, K1), dtype=torch.int32, device=target.device)
    code = load().spec_accept(_ptr(target), _ptr(draft) if K > 0 else None, B, K, _ptr(n_out),
                              _ptr(tok_out), _stream(stream))
    _check(code, "spec_accept")
    return n_out, tok_out


def w8_lmhead_argmax_accept(X, W, scale, draft, out=None, n_out=None, tok_out=None, maxlogit=None, ws=None,
                            stream=None, batch_invariant=False):
    """lm_head argmax of the B*(n+1) rows of X and greedy acceptance of drafts [B][n] in one launch.
    Returns (tokens [B*(n+1)], n_accepted [B], emitted tokens [B][n+1])."""
    import torch
    M, K = X.shape
    V = W.shape[0]
    B, nd = draft.shape
    if out is None:
        out = torch.empty(M, dtype=torch.int32, device=X.device)
    if n_out is None:
        n_out = torch.empty(B, dtype=torch.int32, device=X.device)
    if tok_out is None:
        tok_out = torch.empty((B, nd + 1), dtype=torch.int32, device=X.device)
    if M != B * (nd + 1):
        raise W4VError(ERR_SHAPE, "w8_lmhead_argmax_accept")
    if ws is None:
        ws = workspace(w8_lmhead_argmax_workspace_bytes(M, V), X.device)
    code = load().w8_lmhead_argmax_accept_ex(_ptr(X), _ptr(W), _ptr(scale), B, nd, K, V,
                                             _ptr(draft) if nd > 0 else None, _ptr(out), _ptr(n_out),
                                             _ptr(tok_out), _ptr(maxlogit), _ptr(ws), ws.numel(),
                                             BATCH_INVARIANT if batch_invariant else 0, _stream(stream))
    _check(code, "w8_lmhead_argmax_accept")
    return out, n_out, tok_out


def ngram_draft(context, lengths, n_min: int, n_max: int, K: int, out=None, match=None, ws=None, stream=None):
    """Prompt-lookup drafts on the GPU: context int32 [B][ld], lengths int32 [B] (cuda).
    Returns (drafts int32 [B][K], match length int32 [B])."""
    import torch
    B, ld = context.shape
    if out is None:
        out = torch.empty((B, K), dtype=torch.int32, device=context.device)
    if match is None:
        match = torch.empty(B, dtype=torch.int32, device=context.device)
    if ws is None:
        ws = workspace(load().ngram_draft_workspace_bytes(B), context.device)
    code = load().ngram_draft(_ptr(context), _ptr(lengths), B, ld, int(n_min), int(n_max), int(K),
                              _ptr(out) if K > 0 else None, _ptr(match), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "ngram_draft")
    return out, match


def gdn_verify(state, q, k, v, alpha, beta, out=None, stream=None):
    """Outputs o [B][T][H][dv] (fp16) of the gated delta recurrence over a verify block,
    from the committed fp32 state [B][H][dv][dk]; the state is not written."""
    import torch
    B, H, dv, dk = state.shape
    T = q.shape[1]
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float16, device=state.device)
    code = load().gdn_verify(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), B, T, H, dk, dv,
                             _ptr(out), _stream(stream))
    _check(code, "gdn_verify")
    return out


def gdn_step(state, prev, q, k, v, alpha, beta, out=None, stream=None):
    """Commit the previous block into the fp32 state (prev = (k, v, alpha, beta,
    n_accepted) of that block, or None) and return the outputs o [B][T][H][dv]
    of the current block from the state just committed; one launch."""
    import torch
    B, H, dv, dk = state.shape
    T = q.shape[1]
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float16, device=state.device)
    if prev is None:
        kp = vp = ap = bp = n = None
        T_prev = 0
    else:
        kp, vp, ap, bp, n = prev
        T_prev = kp.shape[1]
    code = load().gdn_step(_ptr(state), _ptr(kp), _ptr(vp), _ptr(ap), _ptr(bp), _ptr(n), T_prev, _ptr(q), _ptr(k),
                           _ptr(v), _ptr(alpha), _ptr(beta), B, T, H, dk, dv, _ptr(out), _stream(stream))
    _check(code, "gdn_step")
    return out


def gdn_commit(state, k, v, alpha, beta, n_accepted, stream=None):
    """Advance the committed state in place by positions 0..n_accepted[b] of the block."""
    B, H, dv, dk = state.shape
    T = k.shape[1]
    code = load().gdn_commit(_ptr(state), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(n_accepted), B, T, H,
                             dk, dv, _stream(stream))
    _check(code, "gdn_commit")
    return state
