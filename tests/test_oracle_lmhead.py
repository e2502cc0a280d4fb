"""Pins for the oracle's int8 lm_head and greedy argmax.

"Efficient LLM Challenge Results", sections 3 and 5: the winning target
unties its lm_head and quantizes it to 8 bits, and decodes at temperature 0.
Reading: int8 symmetric weights with one fp16 scale per vocabulary row,
L[r][v] = s[v] * sum_k X[r][k] W[v][k]; the greedy token is the lowest index
among the maxima, with NaN counted as -inf.
"""
import numpy as np

from conftest import read_golden


def test_one_hot_rows_select_activations(oracle_mod):
    """W[v] = e_{pi(v)}, s = 1: L[r][v] = X[r][pi(v)] exactly (catches a transposed W)."""
    M, K, V = 4, 64, 48
    rng = np.random.default_rng(0)
    pi = rng.integers(0, K, V)
    W = np.zeros((V, K), np.int8)
    W[np.arange(V), pi] = 1
    s = np.ones(V, np.float16)
    X = rng.standard_normal((M, K)).astype(np.float16)
    L = oracle_mod.lmhead_logits(X, W, s)
    assert np.array_equal(L, X.astype(np.float64)[:, pi])


def test_row_scale_and_int8_range(oracle_mod):
    """Weight -127..127 on one k, distinct power-of-two row scales: L = s[v] * w * x."""
    M, K, V = 1, 32, 255
    X = np.zeros((M, K), np.float16)
    X[0, 3] = 1.5
    W = np.zeros((V, K), np.int8)
    W[:, 3] = np.arange(-127, 128)
    s = (2.0 ** -(np.arange(V) % 12)).astype(np.float16)
    L = oracle_mod.lmhead_logits(X, W, s)
    want = s.astype(np.float64) * np.arange(-127, 128) * 1.5
    assert np.array_equal(L[0], want)


def test_argmax_known_by_construction(oracle_mod):
    """One-hot lm_head with unit scales: the greedy token of row r is the v
    whose pi(v) picks the largest activation."""
    M, K, V = 6, 32, 32
    rng = np.random.default_rng(1)
    pi = rng.permutation(K)
    W = np.zeros((V, K), np.int8)
    W[np.arange(V), pi] = 1
    X = rng.standard_normal((M, K)).astype(np.float16)
    L = oracle_mod.lmhead_logits(X, W, np.ones(V, np.float16))
    tok = oracle_mod.argmax(L)
    for r in range(M):
        kbest = int(np.argmax(X[r].astype(np.float64)))
        assert tok[r] == int(np.where(pi == kbest)[0][0])


def _parse_row(field):
    return np.array([float(x) for x in field.split()], np.float32)


def test_argmax_golden_rows(oracle_mod):
    rows = read_golden("argmax_cases.txt")
    assert len(rows) >= 10
    for vals, want in rows:
        row = _parse_row(vals)
        assert oracle_mod.argmax(row.astype(np.float64)) == int(want), vals
        assert oracle_mod.argmax(row) == int(want), vals


def test_argmax_matches_numpy_first_index(oracle_mod):
    """On NaN-free rows numpy.argmax also returns the first maximal index."""
    rng = np.random.default_rng(2)
    L = rng.integers(-5, 5, size=(200, 40)).astype(np.float64)   # many ties
    assert np.array_equal(oracle_mod.argmax(L), np.argmax(L, axis=1))
    L32 = rng.standard_normal((50, 1000)).astype(np.float32)
    assert np.array_equal(oracle_mod.argmax(L32), np.argmax(L32, axis=1))


def test_argmax_rows_matches_full(oracle_mod):
    M, K, V = 7, 128, 300
    rng = np.random.default_rng(3)
    X = rng.standard_normal((M, K)).astype(np.float16)
    W = rng.integers(-127, 128, (V, K), dtype=np.int8)
    s = rng.uniform(1e-3, 5e-3, V).astype(np.float16)
    L = oracle_mod.lmhead_logits(X, W, s)
    rows = np.array([0, 3, 6, 3], np.int32)
    tok, best, second = oracle_mod.lmhead_argmax_rows(X, W, s, rows)
    full = oracle_mod.argmax(L)
    for i, r in enumerate(rows):
        assert tok[i] == full[r]
        srt = np.sort(L[r])
        assert best[i] == srt[-1] and second[i] == srt[-2]


def test_argmax_rows_ties_go_to_the_lowest_index(oracle_mod):
    """Vocabulary rows copied with their scale give exactly equal logits: the
    row-sampled argmax takes the first copy, and the second-best logit equals
    the best one (known by construction, no full logits needed)."""
    M, K, V = 3, 64, 40
    rng = np.random.default_rng(4)
    X = rng.standard_normal((M, K)).astype(np.float16)
    W = rng.integers(-127, 128, (V, K), dtype=np.int8)
    s = rng.uniform(1e-3, 5e-3, V).astype(np.float16)
    tok0, _, _ = oracle_mod.lmhead_argmax_rows(X, W, s, np.arange(M, dtype=np.int32))
    # copy each row's winner to two other slots, then also to the first slot
    for r in range(M):
        W2, s2 = W.copy(), s.copy()
        w = int(tok0[r])
        copies = [d for d in (V - 1, V - 7) if d != w]
        for dst in copies:
            W2[dst], s2[dst] = W[w], s[w]
        tok, best, second = oracle_mod.lmhead_argmax_rows(X, W2, s2, np.array([r], np.int32))
        assert tok[0] == min([w] + copies) and second[0] == best[0]
        W2[0], s2[0] = W[w], s[w]
        tok, best, second = oracle_mod.lmhead_argmax_rows(X, W2, s2, np.array([r], np.int32))
        assert tok[0] == 0 and second[0] == best[0]
