"""Toy autoregressive W4A16 target for the greedy speculative-decoding invariant.

Test infrastructure (see the package docstring): only tests and the
benchmark's CPU leg use it.

"Efficient LLM Challenge Results" (AdaptFM @ ICML 2026), section 3
"Speculative decoding did the heavy lifting", states that under greedy
verification speculative decoding leaves the output unchanged whatever the
drafts are (one entry calls it bit-exact regardless of draft quality), and
that drafts padded with -1 sentinels stay lossless because a padded position
is accepted only when it equals the verifier's own greedy token.  This module
builds the smallest real model on which that can be checked token for token:

  * embedding E (fp16 [V][H]); the input at position i is
    x_i = E[t_i] + mean(E[t_0..t_i])  (context dependence without attention);
  * L residual MLP layers  h += down(silu(gate(r)) * up(r)),  r = rms(h),
    with gate/up fused into one W4A16 (group 128) projection H -> 2H and down
    a W4A16 projection H -> H; every projection input is rounded to fp16,
    as W4A16 takes fp16 activations;
  * a final rms, the int8 per-row-scaled lm_head, and the greedy argmax.

Without a recurrent layer each position is a function of the tokens up to it
only, so rolling back rejected draft positions is just dropping them.  The
optional gated-delta layer (first, before the MLPs) adds what the pages warn
about: most of the target's layers are Gated DeltaNet, whose recurrent state
a rejected draft must not touch ("Efficient LLM Challenge Results", section
3, runner-up paragraph; "DFlash K=15 for Qwen3.5-4B on a single A10G", "What
transfers").  Per head (dk = dv = 128), from r = rms(h): a W4A16 q|k|v
projection, q and k scaled to unit length, alpha = sigmoid(2 + wa.r),
beta = sigmoid(wb.r), the recurrence of oracle_gdn_recurrence, and the heads'
outputs through a W4A16 projection added to h.  Greedy decoding recomputes
the state from the first token every step (the definition); speculative
decoding keeps a committed state, verifies K+1 positions from it without
committing, and then commits only the accepted prefix (positions 0..n of the
block), which is what keeps it equal to greedy decoding.  All other
arithmetic is double precision, through the C oracle's GEMM, lm_head, argmax
and recurrence.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Sequence

import numpy as np

from . import argmax, dequant_w4, gdn_recurrence, lmhead_logits, matmul_dequantized, spec_accept

RMS_EPS = 1e-6


@dataclass
class ToyWeights:
    E: np.ndarray                 # fp16 [V][H]
    layers: list                  # [(q_gu [2H][H], s_gu [H/128][2H], q_d [H][H], s_d [H/128][H])]
    W8: np.ndarray                # int8 [V][H]
    s8: np.ndarray                # fp16 [V]
    gdn: tuple | None = None      # (q_qkv [3H][H], s_qkv, q_o [H][H], s_o, wa [heads][H], wb [heads][H])

    def dequantized(self):
        """Per layer (W_gate_up, W_down) dequantized once by the oracle and cached."""
        if getattr(self, "_deq", None) is None:
            self._deq = [(dequant_w4(q_gu, s_gu), dequant_w4(q_d, s_d))
                         for (q_gu, s_gu, q_d, s_d) in self.layers]
        return self._deq

    def gdn_dequantized(self):
        if getattr(self, "_gdn_deq", None) is None:
            q_qkv, s_qkv, q_o, s_o, wa, wb = self.gdn
            self._gdn_deq = (dequant_w4(q_qkv, s_qkv), dequant_w4(q_o, s_o),
                             wa.astype(np.float64), wb.astype(np.float64))
        return self._gdn_deq

    @property
    def heads(self) -> int:
        return 0 if self.gdn is None else self.gdn[4].shape[0]

    def zero_state(self) -> np.ndarray:
        d = self.H // self.heads
        return np.zeros((self.heads, d, d), np.float64)

    @property
    def V(self) -> int:
        return self.E.shape[0]

    @property
    def H(self) -> int:
        return self.E.shape[1]


def _rms(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + RMS_EPS)


def _silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def _inputs(w: ToyWeights, tokens: Sequence[int], positions: Sequence[int]) -> np.ndarray:
    """x_p = E[t_p] + mean(E[t_0..t_p]) for each requested position p."""
    E = w.E.astype(np.float64)
    emb = E[np.asarray(tokens, dtype=np.int64)]
    csum = np.cumsum(emb, axis=0)
    pos = np.asarray(positions, dtype=np.int64)
    return emb[pos] + csum[pos] / (pos[:, None] + 1.0)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def gdn_layer(w: ToyWeights, h: np.ndarray, S: np.ndarray):
    """The gated-delta layer over consecutive positions (rows of h) starting from
    state S: returns (h + its output, the state after the last row)."""
    W_qkv, W_o, wa, wb = w.gdn_dequantized()
    H, nh = w.H, w.heads
    d = H // nh
    r = _rms(h).astype(np.float16)
    qkv = matmul_dequantized(r, W_qkv)
    T = h.shape[0]
    q = qkv[:, :H].reshape(T, nh, d)
    k = qkv[:, H:2 * H].reshape(T, nh, d)
    v = qkv[:, 2 * H:].reshape(T, nh, d)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    rd = r.astype(np.float64)
    alpha = _sigmoid(2.0 + rd @ wa.T)
    beta = _sigmoid(rd @ wb.T)
    o, S_out = gdn_recurrence(S, q, k, v, alpha, beta)
    return h + matmul_dequantized(o.reshape(T, H).astype(np.float16), W_o), S_out


def hidden_at(w: ToyWeights, tokens: Sequence[int], positions: Sequence[int], state=None) -> np.ndarray:
    """Final normalised hidden rows (fp16 [len(positions)][H]) fed to the lm_head.

    With a gated-delta layer the positions must be consecutive; `state` is the
    recurrent state before the first of them (None: recomputed from the first
    token, the definition)."""
    H = w.H
    if w.gdn is not None:
        p0 = int(positions[0])
        assert list(positions) == list(range(p0, p0 + len(positions)))
        if state is None:
            state = prefix_state(w, tokens, p0)
        h, _ = gdn_layer(w, _inputs(w, tokens, positions), state)
    else:
        h = _inputs(w, tokens, positions)
    for (w_gu, w_d) in w.dequantized():
        r = _rms(h).astype(np.float16)
        gu = matmul_dequantized(r, w_gu)
        a = (_silu(gu[:, :H]) * gu[:, H:]).astype(np.float16)
        h = h + matmul_dequantized(a, w_d)
    return _rms(h).astype(np.float16)


def prefix_state(w: ToyWeights, tokens: Sequence[int], n: int) -> np.ndarray:
    """Recurrent state after positions 0..n-1, from the zero state."""
    S = w.zero_state()
    if n > 0:
        _, S = gdn_layer(w, _inputs(w, tokens, list(range(n))), S)
    return S


def advance_state(w: ToyWeights, tokens: Sequence[int], p0: int, count: int, S: np.ndarray) -> np.ndarray:
    """State after positions p0 .. p0+count-1, from the state S before p0."""
    if count <= 0:
        return S
    _, S = gdn_layer(w, _inputs(w, tokens, list(range(p0, p0 + count))), S)
    return S


def logits_at(w: ToyWeights, tokens: Sequence[int], positions: Sequence[int], state=None) -> np.ndarray:
    """Target logits (double [len(positions)][V]) for the given sequence positions."""
    return lmhead_logits(hidden_at(w, tokens, positions, state), w.W8, w.s8)


def greedy_decode(w: ToyWeights, prompt: Sequence[int], n_new: int) -> List[int]:
    """Plain greedy decoding: one position per step (M = 1)."""
    ctx = list(prompt)
    out: List[int] = []
    while len(out) < n_new:
        tok = int(argmax(logits_at(w, ctx, [len(ctx) - 1]))[0])
        ctx.append(tok)
        out.append(tok)
    return out


Drafter = Callable[[List[int], int], List[int]]


def spec_decode(w: ToyWeights, prompt: Sequence[int], n_new: int, K: int,
                drafter: Drafter, stats: dict | None = None, commit: str = "accepted") -> List[int]:
    """Greedy speculative decoding with a K-token drafter.

    Each step verifies K+1 positions in one call: position j sees the context
    plus drafts d[0..j-1] and yields the target's greedy token t[j].  The
    accepted prefix n and the emitted tokens d[0..n-1] + t[n] come from the
    oracle's acceptance rule.  A sentinel draft (negative) is fed to the
    model as token 0; no position after it can be accepted, and t[n] for the
    first sentinel position n does not depend on that placeholder.

    With a gated-delta layer the recurrent state of positions 0..len(ctx)-2
    is kept committed; the K+1 block is verified from it without committing,
    and then positions 0..n of the block (the last context token and the n
    accepted drafts) are committed.  `commit` exists for the test that shows
    the invariant catches the failures the pages describe: "all" also
    commits the rejected positions, "none" never advances the state (a
    stale state).
    """
    ctx = list(prompt)
    out: List[int] = []
    steps = 0
    accepted = 0
    S = prefix_state(w, ctx, len(ctx) - 1) if w.gdn is not None else None
    while len(out) < n_new:
        d = list(drafter(list(ctx), K)) if K > 0 else []
        assert len(d) == K
        seq = ctx + [x if x >= 0 else 0 for x in d]
        p0 = len(ctx) - 1
        positions = [p0 + j for j in range(K + 1)]
        t = argmax(logits_at(w, seq, positions, S)).astype(np.int32)
        n, tok = spec_accept(t[None, :], np.asarray(d, np.int32).reshape(1, K))
        n = int(n[0])
        emitted = [int(x) for x in tok[0, : n + 1]]
        if S is not None:
            count = {"accepted": n + 1, "all": K + 1, "none": 0}[commit]
            S = advance_state(w, seq, p0, count, S)
        ctx.extend(emitted)
        out.extend(emitted)
        steps += 1
        accepted += n
    if stats is not None:
        stats["steps"] = steps
        stats["accepted"] = accepted
    return out[:n_new]
