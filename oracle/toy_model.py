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

Each position is a function of the tokens up to it only, so rolling back
rejected draft positions is just dropping them.  All other arithmetic is
double precision, through the C oracle's GEMM, lm_head and argmax.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Sequence

import numpy as np

from . import argmax, dequant_w4, lmhead_logits, matmul_dequantized, spec_accept

RMS_EPS = 1e-6


@dataclass
class ToyWeights:
    E: np.ndarray                 # fp16 [V][H]
    layers: list                  # [(q_gu [2H][H], s_gu [H/128][2H], q_d [H][H], s_d [H/128][H])]
    W8: np.ndarray                # int8 [V][H]
    s8: np.ndarray                # fp16 [V]

    def dequantized(self):
        """Per layer (W_gate_up, W_down) dequantized once by the oracle and cached."""
        if getattr(self, "_deq", None) is None:
            self._deq = [(dequant_w4(q_gu, s_gu), dequant_w4(q_d, s_d))
                         for (q_gu, s_gu, q_d, s_d) in self.layers]
        return self._deq

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


def hidden_at(w: ToyWeights, tokens: Sequence[int], positions: Sequence[int]) -> np.ndarray:
    """Final normalised hidden rows (fp16 [len(positions)][H]) fed to the lm_head."""
    H = w.H
    h = _inputs(w, tokens, positions)
    for (w_gu, w_d) in w.dequantized():
        r = _rms(h).astype(np.float16)
        gu = matmul_dequantized(r, w_gu)
        a = (_silu(gu[:, :H]) * gu[:, H:]).astype(np.float16)
        h = h + matmul_dequantized(a, w_d)
    return _rms(h).astype(np.float16)


def logits_at(w: ToyWeights, tokens: Sequence[int], positions: Sequence[int]) -> np.ndarray:
    """Target logits (double [len(positions)][V]) for the given sequence positions."""
    return lmhead_logits(hidden_at(w, tokens, positions), w.W8, w.s8)


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
                drafter: Drafter, stats: dict | None = None) -> List[int]:
    """Greedy speculative decoding with a K-token drafter.

    Each step verifies K+1 positions in one call: position j sees the context
    plus drafts d[0..j-1] and yields the target's greedy token t[j].  The
    accepted prefix n and the emitted tokens d[0..n-1] + t[n] come from the
    oracle's acceptance rule.  A sentinel draft (negative) is fed to the
    model as token 0; no position after it can be accepted, and t[n] for the
    first sentinel position n does not depend on that placeholder.
    """
    ctx = list(prompt)
    out: List[int] = []
    steps = 0
    accepted = 0
    while len(out) < n_new:
        d = list(drafter(list(ctx), K)) if K > 0 else []
        assert len(d) == K
        seq = ctx + [x if x >= 0 else 0 for x in d]
        positions = [len(ctx) - 1 + j for j in range(K + 1)]
        t = argmax(logits_at(w, seq, positions)).astype(np.int32)
        n, tok = spec_accept(t[None, :], np.asarray(d, np.int32).reshape(1, K))
        n = int(n[0])
        emitted = [int(x) for x in tok[0, : n + 1]]
        ctx.extend(emitted)
        out.extend(emitted)
        steps += 1
        accepted += n
    if stats is not None:
        stats["steps"] = steps
        stats["accepted"] = accepted
    return out[:n_new]
