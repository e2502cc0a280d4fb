"""Pins for the oracle's greedy acceptance rule.

The rule comes from "Efficient LLM Challenge Results", section 3: keep the
longest draft prefix the target would itself have produced; a -1 padding
sentinel is accepted only if it equals the target's greedy token, which it
never does.  The pins are hand-worked cases (tests/golden/accept_cases.txt),
an exhaustive enumeration on tiny vocabularies checked against the
properties that characterise the accepted prefix, and the invariant that
speculative decoding with this rule reproduces greedy decoding exactly.
"""
import itertools

import numpy as np
import pytest

from conftest import read_golden


def _ints(field):
    return [int(x) for x in field.split()] if field.strip() else []


def test_golden_cases(oracle_mod):
    rows = read_golden("accept_cases.txt")
    assert len(rows) >= 10
    for d, t, n, emitted in rows:
        d, t, n, emitted = _ints(d), _ints(t), int(n), _ints(emitted)
        assert len(t) == len(d) + 1
        got_n, tok = oracle_mod.spec_accept(np.asarray(t, np.int32), np.asarray(d, np.int32))
        assert got_n == n, (d, t)
        assert list(tok[: n + 1]) == emitted, (d, t)
        assert all(x == -1 for x in tok[n + 1:])


@pytest.mark.parametrize("V,K", [(1, 3), (2, 3), (3, 2), (2, 4), (3, 3)])
def test_exhaustive_tiny_vocab(oracle_mod, V, K):
    """All (target, draft) pairs, drafts over {-1} + [0, V): the accepted prefix
    must (a) agree with the target, (b) stop at the first disagreement or at
    K, (c) never include a sentinel, and (d) emit exactly the target's own
    tokens t[0..n]."""
    targets = list(itertools.product(range(V), repeat=K + 1))
    drafts = list(itertools.product(range(-1, V), repeat=K))
    T = np.array([t for t in targets for _ in drafts], np.int32)
    D = np.array([d for _ in targets for d in drafts], np.int32).reshape(len(T), K)
    n, tok = oracle_mod.spec_accept(T, D)
    for i in range(len(T)):
        t, d, ni = T[i], D[i], int(n[i])
        assert 0 <= ni <= K
        assert all(d[j] == t[j] for j in range(ni))                  # (a)
        assert ni == K or d[ni] != t[ni] or d[ni] < 0                  # (b)
        assert all(d[j] >= 0 for j in range(ni))                       # (c)
        assert list(tok[i, : ni + 1]) == list(t[: ni + 1])             # (d)
        assert all(x == -1 for x in tok[i, ni + 1:])


def _markov_greedy(table, start, n):
    out, cur = [], start
    for _ in range(n):
        cur = int(table[cur])
        out.append(cur)
    return out


@pytest.mark.parametrize("seed", range(5))
def test_spec_equals_greedy_markov_target(oracle_mod, seed):
    """With a deterministic next-token function standing in for the target,
    speculative decoding with any drafts emits the greedy sequence."""
    rng = np.random.default_rng(seed)
    V, K, n_new = 7, 5, 40
    table = rng.integers(0, V, size=V)
    start = int(rng.integers(0, V))
    want = _markov_greedy(table, start, n_new)
    for mode in ("random", "perfect", "sentinel", "mixed"):
        ctx, out = [start], []
        while len(out) < n_new:
            truth = _markov_greedy(table, ctx[-1], K)
            if mode == "random":
                d = list(rng.integers(-1, V, size=K))
            elif mode == "perfect":
                d = truth
            elif mode == "sentinel":
                d = [-1] * K
            else:
                j = int(rng.integers(0, K + 1))
                d = truth[:j] + list(rng.integers(-1, V, size=K - j))
            # target's greedy token after each verify position: position j sees ctx + d[:j]
            prev = [ctx[-1]] + [x if x >= 0 else 0 for x in d]
            t = [int(table[p]) for p in prev]
            n, tok = oracle_mod.spec_accept(np.asarray(t, np.int32), np.asarray(d, np.int32))
            emitted = list(tok[: n + 1])
            ctx += emitted
            out += emitted
        assert out[:n_new] == want, mode


def test_accepted_length_distribution(oracle_mod):
    """Drafts that match each target token independently with probability a
    give P(n >= j) = a**j (the prefix survives j independent matches)."""
    from speculative_decoding_verify_w4a16_gb300 import inputs
    B, K, V = 20000, 6, 1000
    r = np.random.default_rng(123)
    t = r.integers(0, V, size=(B, K + 1)).astype(np.int32)
    for a in (0.25, 0.5, 0.9):
        d = inputs.drafts_alpha(7, t, V, a)
        n, _ = oracle_mod.spec_accept(t, d)
        for j in range(1, K + 1):
            p = float(np.mean(n >= j))
            sd = np.sqrt(a ** j * (1 - a ** j) / B)
            assert abs(p - a ** j) <= 5 * sd + 1e-9, (a, j, p)
