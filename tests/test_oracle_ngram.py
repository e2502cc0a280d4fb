"""The oracle's prompt-lookup (n-gram) drafter against hand-worked cases and
against the definition checked by enumeration.

"Efficient LLM Challenge Results", section 3 (table of drafting methods):
n-gram / prompt-lookup drafting copies spans from the prompt with no
auxiliary model.  The reading (longest n-gram first, latest earlier
occurrence, -1 padding where the context ends) is worked by hand in
tests/golden/ngram_cases.txt; every case there was derived on paper.
"""
import itertools

import numpy as np
import pytest

from conftest import read_golden


def _ints(field):
    return [int(x) for x in field.split()] if field.strip() else []


def test_golden_cases(oracle_mod):
    rows = read_golden("ngram_cases.txt")
    assert len(rows) >= 12
    for ctx, params, drafts, match in rows:
        c = np.array(_ints(ctx), np.int32)
        n_min, n_max, K = _ints(params)
        d, m = oracle_mod.ngram_draft(c.reshape(1, -1) if c.size else np.zeros((1, 1), np.int32),
                                      [c.size], n_min, n_max, K)
        assert list(d[0]) == _ints(drafts), ctx
        assert int(m[0]) == int(match), ctx


def _properties_hold(c, n_min, n_max, K, d, m):
    """The result satisfies the definition: m is the largest n in [n_min, n_max]
    whose suffix n-gram occurs at some start p with p + n <= L - 1, d copies
    what followed the latest such p (padded with -1), and m == 0 means none."""
    L = len(c)
    occ = {n: [p for p in range(0, L - n) if c[p:p + n] == c[L - n:]]
           for n in range(n_min, n_max + 1) if 1 <= n <= L - 1}
    ns = [n for n, ps in occ.items() if ps]
    if not ns:
        return m == 0 and d == [-1] * K
    n = max(ns)
    p = max(occ[n])
    want = (c[p + n:p + n + K] + [-1] * K)[:K]
    return m == n and d == want


def test_enumeration_small_alphabet(oracle_mod):
    """Every context of length 0..7 over three tokens, n in [1, 3], K = 4."""
    ctxs = []
    for L in range(0, 8):
        for c in itertools.product(range(3), repeat=L):
            ctxs.append(list(c))
    B = len(ctxs)
    ld = 7
    arr = np.full((B, ld), 99, np.int32)
    lens = np.zeros(B, np.int32)
    for i, c in enumerate(ctxs):
        arr[i, :len(c)] = c
        lens[i] = len(c)
    for n_min, n_max in ((1, 3), (2, 3), (1, 1), (3, 6)):
        d, m = oracle_mod.ngram_draft(arr, lens, n_min, n_max, 4)
        for i, c in enumerate(ctxs):
            assert _properties_hold(c, n_min, n_max, 4, list(d[i]), int(m[i])), (c, n_min, n_max)


def test_rows_are_independent_of_padding(oracle_mod):
    """Tokens past a row's length never influence its drafts."""
    rng = np.random.default_rng(3)
    ctx = rng.integers(0, 5, size=(6, 40)).astype(np.int32)
    lens = np.array([0, 1, 7, 20, 39, 40], np.int32)
    d1, m1 = oracle_mod.ngram_draft(ctx, lens, 1, 4, 6)
    ctx2 = ctx.copy()
    for b, L in enumerate(lens):
        ctx2[b, L:] = 4 - ctx2[b, L:]
    d2, m2 = oracle_mod.ngram_draft(ctx2, lens, 1, 4, 6)
    assert np.array_equal(d1, d2) and np.array_equal(m1, m2)


@pytest.mark.parametrize("period", [1, 2, 5, 13])
def test_periodic_context_continues_the_period(oracle_mod, period):
    """A context that repeats a block of `period` distinct tokens is drafted
    as the block's continuation: the latest earlier occurrence of the suffix
    n-gram is exactly one period back."""
    block = list(range(100, 100 + period))
    L = 4 * period + 3
    c = (block * 10)[:L]
    K = 2 * period + 1
    d, m = oracle_mod.ngram_draft(np.array(c, np.int32), None, 1, 3, K)
    assert m == 3
    p = L - period - m                       # start of the occurrence one period back
    want = (c[p + m:] + [-1] * K)[:K]
    assert list(d) == want
