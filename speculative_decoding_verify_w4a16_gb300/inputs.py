"""Seeded synthetic inputs for the verify step.

This module holds no arithmetic of the method: it only draws random arrays
(numpy PCG64, identical on every platform) with the shapes and value
distributions of the workloads, and builds drafts from target tokens that the
caller supplies.  Both the CUDA path and the CPU oracle are fed from here.

Value recipes:
  * int4 weight codes q ~ U{0..15}, logical layout [N][K] (one code per byte);
  * group scales s ~ U[0.005, 0.02] rounded to fp16, layout [K/128][N];
  * activations ~ N(0, 1) rounded to fp16, layout [M][K];
  * int8 lm_head W8 ~ U{-127..127}, layout [V][K]; row scales ~ U[1e-3, 5e-3]
    rounded to fp16.
Every array is drawn from its own stream keyed by (seed, tag...), so a
layer's weights can be regenerated without drawing the ones before it.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass
from typing import Dict, List, Tuple

import numpy as np

GROUP = 128
ALPHAS = (0.0, 0.25, 0.5, 0.75, 0.9, 1.0)


def _key(tag) -> int:
    if isinstance(tag, str):
        return zlib.crc32(tag.encode())
    return int(tag)


def rng(seed: int, *tags) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed)] + [_key(t) for t in tags])))


def w4_codes(seed: int, N: int, K: int, *tags) -> np.ndarray:
    return rng(seed, "q", N, K, *tags).integers(0, 16, size=(N, K), dtype=np.uint8)


def w4_scales(seed: int, N: int, K: int, *tags, group: int = GROUP) -> np.ndarray:
    r = rng(seed, "s", N, K, *tags)
    return r.uniform(0.005, 0.02, size=(K // group, N)).astype(np.float16)


def w4_zeros(seed: int, N: int, K: int, *tags, group: int = GROUP) -> np.ndarray:
    """Asymmetric (AWQ-style) zero points, U{0..15}, layout [K/G][N]."""
    return rng(seed, "z", N, K, *tags).integers(0, 16, size=(K // group, N), dtype=np.uint8)


def activations(seed: int, M: int, K: int, *tags) -> np.ndarray:
    r = rng(seed, "a", M, K, *tags)
    return r.standard_normal(size=(M, K), dtype=np.float32).astype(np.float16)


def lmhead_weights(seed: int, V: int, K: int, *tags) -> Tuple[np.ndarray, np.ndarray]:
    W8 = rng(seed, "w8", V, K, *tags).integers(-127, 128, size=(V, K), dtype=np.int8)
    s8 = rng(seed, "s8", V, *tags).uniform(1e-3, 5e-3, size=V).astype(np.float16)
    return W8, s8


def alpha_for_seed(seed: int) -> float:
    """Per-seed draft acceptance rate, drawn from a fixed menu."""
    return float(ALPHAS[int(rng(seed, "alpha").integers(0, len(ALPHAS)))])


def drafts_half_match(seed: int, target: np.ndarray, V: int) -> np.ndarray:
    """K drafts uniform in [0, V), then floor(K/2) seeded positions forced to equal target."""
    t = np.asarray(target, np.int32)
    K = t.shape[-1] - 1
    r = rng(seed, "dhalf", K, V)
    d = r.integers(0, V, size=K, dtype=np.int64).astype(np.int32)
    if K > 0:
        pos = r.choice(K, size=K // 2, replace=False)
        d[pos] = t[pos]
    return d


def drafts_alpha(seed: int, target: np.ndarray, V: int, alpha: float | None = None,
                 *tags) -> np.ndarray:
    """Per position i: d[i] = t[i] with probability alpha, else a uniform token != t[i].

    target int32 [..., K+1] -> drafts int32 [..., K].
    """
    t = np.asarray(target, np.int32)
    K = t.shape[-1] - 1
    a = alpha_for_seed(seed) if alpha is None else float(alpha)
    r = rng(seed, "dalpha", K, V, *tags)
    shape = t.shape[:-1] + (K,)
    hit = r.random(size=shape) < a
    other = r.integers(0, V - 1, size=shape, dtype=np.int64)
    tk = t[..., :K].astype(np.int64)
    wrong = other + (other >= tk)          # uniform over [0, V) without t[i]
    return np.where(hit, tk, wrong).astype(np.int32)


def drafts_padded(seed: int, target: np.ndarray, V: int, alpha: float | None = None,
                  *tags) -> Tuple[np.ndarray, np.ndarray]:
    """Constant-K drafts: a seeded real length L in [0, K], positions >= L set to -1."""
    t = np.asarray(target, np.int32)
    K = t.shape[-1] - 1
    d = drafts_alpha(seed, t, V, alpha, "pad", *tags)
    L = rng(seed, "dlen", K, *tags).integers(0, K + 1, size=t.shape[:-1])
    idx = np.arange(K)
    d = np.where(idx < np.asarray(L)[..., None], d, -1).astype(np.int32)
    return d, np.asarray(L)


# ----------------------------------------------------------------- configs --
H_4B = 2560
I_4B = 9728
V_4B = 151936


@dataclass(frozen=True)
class Proj:
    name: str
    N: int
    K: int


LAYER_PROJS: Tuple[Proj, ...] = (
    Proj("qkv", 3 * H_4B, H_4B),
    Proj("o", H_4B, H_4B),
    Proj("gate_up", 2 * I_4B, H_4B),
    Proj("down", H_4B, I_4B),
)

CONFIGS: Dict[str, dict] = {
    "cfg0": dict(desc="tiny verify: one W4A16 linear 256->512 at M=16, int8 lm_head 256->1024, K=15",
                 M=16, projs=(Proj("linear", 512, 256),), V=1024, H=256, K_draft=15, B=1),
    "cfg1": dict(desc="one 4B-shaped layer set (qkv, o, gate_up, down) at M=16 + int8 lm_head 2560->151936, K=15",
                 M=16, projs=LAYER_PROJS, V=V_4B, H=H_4B, K_draft=15, B=1),
    "cfg2": dict(desc="36-layer stack of the layer set, M in {1,2,4,8,16,21}, K=M-1 (K=20 padded with -1)",
                 layers=36, M_sweep=(1, 2, 4, 8, 16, 21), projs=LAYER_PROJS, V=V_4B, H=H_4B, B=1),
    "cfg3": dict(desc="prefill layer set at M=2048, lm_head on the last row",
                 M=2048, projs=LAYER_PROJS, V=V_4B, H=H_4B, lm_rows=1),
    "cfg4": dict(desc="prefill layer set at M=8192; lm_head verify of 8 sequences x 16 positions (M=128), K=15",
                 M=8192, projs=LAYER_PROJS, V=V_4B, H=H_4B, B=8, K_draft=15),
}


def layer_weights(seed: int, layer: int, proj: Proj):
    """(codes [N][K], scales [K/128][N]) for one projection of one layer."""
    return (w4_codes(seed, proj.N, proj.K, layer, proj.name),
            w4_scales(seed, proj.N, proj.K, layer, proj.name))


def toy_model_arrays(seed: int, V: int = 64, H: int = 256, layers: int = 2):
    """Random weights for the toy autoregressive model: E, per-layer (gate_up, down), lm_head."""
    E = rng(seed, "toyE", V, H).standard_normal(size=(V, H), dtype=np.float32).astype(np.float16)
    lay = []
    for l in range(layers):
        q_gu = w4_codes(seed, 2 * H, H, "toy", l, "gu")
        s_gu = w4_scales(seed, 2 * H, H, "toy", l, "gu")
        q_d = w4_codes(seed, H, H, "toy", l, "d")
        s_d = w4_scales(seed, H, H, "toy", l, "d")
        lay.append((q_gu, s_gu, q_d, s_d))
    W8, s8 = lmhead_weights(seed, V, H, "toy")
    return E, lay, W8, s8


def random_tokens(seed: int, n: int, V: int, *tags) -> List[int]:
    return [int(x) for x in rng(seed, "tok", n, V, *tags).integers(0, V, size=n)]


def ngram_contexts(seed: int, B: int, ld: int, V: int, *tags, copy_prob: float = 0.5,
                   ragged: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """Prompt-like token contexts for prompt-lookup drafting: int32 [B][ld] and
    lengths [B].  Each row grows by spans of 4..32 tokens that are, with
    probability copy_prob, copies of an earlier span of the same row (the
    repeated passages prompt lookup feeds on), else fresh uniform tokens.
    Ragged lengths are uniform in [ld/2, ld]; tokens past a row's length are
    uniform filler."""
    r = rng(seed, "ngctx", B, ld, V, *tags)
    ctx = r.integers(0, V, size=(B, ld), dtype=np.int64).astype(np.int32)
    if ragged:
        lens = r.integers(ld // 2, ld + 1, size=B).astype(np.int32)
    else:
        lens = np.full(B, ld, np.int32)
    for b in range(B):
        L = int(lens[b])
        pos = min(L, int(r.integers(4, 33)))
        while pos < L:
            n = min(L - pos, int(r.integers(4, 33)))
            if pos >= 8 and r.random() < copy_prob:
                src = int(r.integers(0, pos - 4))
                for i in range(n):           # may overlap its own output, like a repeat
                    ctx[b, pos + i] = ctx[b, src + i]
            pos += n
    return ctx, lens


def toy_gdn_arrays(seed: int, H: int = 256, heads: int = 2):
    """Weights of the toy model's gated-delta layer: a fused W4A16 q|k|v
    projection H -> 3H, a W4A16 output projection H -> H, and fp16 gate
    vectors [heads][H] for the decay (alpha) and the write strength (beta)."""
    q_qkv = w4_codes(seed, 3 * H, H, "toy-gdn", "qkv")
    s_qkv = w4_scales(seed, 3 * H, H, "toy-gdn", "qkv")
    q_o = w4_codes(seed, H, H, "toy-gdn", "o")
    s_o = w4_scales(seed, H, H, "toy-gdn", "o")
    r = rng(seed, "toy-gdn-gates", heads, H)
    wa = (r.standard_normal(size=(heads, H)) / np.sqrt(H)).astype(np.float16)
    wb = (r.standard_normal(size=(heads, H)) / np.sqrt(H)).astype(np.float16)
    return q_qkv, s_qkv, q_o, s_o, wa, wb
