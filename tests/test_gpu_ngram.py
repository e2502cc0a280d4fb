"""ngram_draft on the GPU against the oracle, bit for bit ("Efficient LLM
Challenge Results", section 3, table of drafting methods: n-gram /
prompt-lookup drafting copies spans from the prompt).  Drafts and match
lengths are integers, so the bar is exact equality: on the hand-worked
golden cases, on prompt-like synthetic contexts with ragged lengths, on
contexts long enough to split over many CTAs, and on the degenerate ones
(empty, one token, no match, overlapping and periodic continuations)."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from helpers import to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _ints(field):
    return [int(x) for x in field.split()] if field.strip() else []


def _both(w4v_mod, oracle_mod, gpu, ctx, lens, n_min, n_max, K):
    d_o, m_o = oracle_mod.ngram_draft(ctx, lens, n_min, n_max, K)
    d_g, m_g = w4v_mod.ngram_draft(to_dev(ctx, gpu), to_dev(np.asarray(lens, np.int32), gpu), n_min, n_max, K)
    torch.cuda.synchronize()
    assert np.array_equal(d_g.cpu().numpy(), d_o)
    assert np.array_equal(m_g.cpu().numpy(), m_o)
    assert w4v_mod.get_status() == 0
    return m_o


def test_golden_cases_gpu(w4v_mod, gpu, oracle_mod):
    for ctx, params, drafts, match in read_golden("ngram_cases.txt"):
        c = _ints(ctx)
        n_min, n_max, K = _ints(params)
        arr = np.array([c + [0]] if c else [[0]], np.int32)
        d, m = w4v_mod.ngram_draft(to_dev(arr, gpu), to_dev(np.array([len(c)], np.int32), gpu), n_min, n_max, K)
        torch.cuda.synchronize()
        assert list(d.cpu().numpy()[0]) == _ints(drafts), ctx
        assert int(m.cpu()[0]) == int(match), ctx


@pytest.mark.parametrize("B,ld,V,n_min,n_max,K", [
    (8, 4096, 151936, 1, 4, 23),     # the n-gram entry's K = 23, 4B vocabulary
    (8, 4096, 151936, 2, 8, 15),
    (3, 300, 50, 1, 3, 20),          # small vocabulary: many short matches
    (16, 1000, 7, 1, 64, 32),        # tiny vocabulary, longest n-grams
    (1, 70000, 1000, 1, 5, 128),     # one long row over many CTAs
    (4, 9000, 151936, 3, 3, 1),
])
def test_synthetic_contexts(w4v_mod, gpu, oracle_mod, B, ld, V, n_min, n_max, K):
    ctx, lens = inputs.ngram_contexts(B + ld, B, ld, V, "gpu")
    m = _both(w4v_mod, oracle_mod, gpu, ctx, lens, n_min, n_max, K)
    if V > 1000 and n_min == 1:
        assert np.any(m > 0)          # the copied spans are found


def test_degenerate_rows(w4v_mod, gpu, oracle_mod):
    """Lengths 0, 1, 2, a row without any repeat, an all-equal row, a
    period-3 row, a row whose only match is at the very start, and
    out-of-range lengths (clamped to [0, ld])."""
    ld = 64
    rows, lens = [], []
    def add(tokens, L=None):
        r = (list(tokens) + [0] * ld)[:ld]
        rows.append(r)
        lens.append(len(tokens) if L is None else L)
    add([])
    add([5])
    add([5, 5])
    add(list(range(100, 164)))
    add([9] * 64)
    add([1, 2, 3] * 21 + [1])
    add([7, 8] + list(range(200, 260)) + [7, 8])
    add(list(range(10)) * 7, L=-5)
    add([4, 5, 4, 5] * 16, L=1000)
    ctx = np.array(rows, np.int32)
    lens_c = np.clip(np.array(lens), 0, ld).astype(np.int32)
    d_o, m_o = oracle_mod.ngram_draft(ctx, lens_c, 1, 6, 10)
    d_g, m_g = w4v_mod.ngram_draft(to_dev(ctx, gpu), to_dev(np.array(lens, np.int32), gpu), 1, 6, 10)
    torch.cuda.synchronize()
    assert np.array_equal(d_g.cpu().numpy(), d_o)
    assert np.array_equal(m_g.cpu().numpy(), m_o)
    assert list(m_o[:4]) == [0, 0, 1, 0]


def test_workspace_left_zeroed_and_graph_replay(w4v_mod, gpu, oracle_mod):
    B, ld, V = 8, 5000, 1000
    ctx, lens = inputs.ngram_contexts(3, B, ld, V, "graph")
    d_o, m_o = oracle_mod.ngram_draft(ctx, lens, 1, 4, 23)
    c, l = to_dev(ctx, gpu), to_dev(lens, gpu)
    ws = w4v_mod.workspace(w4v_mod.load().ngram_draft_workspace_bytes(B), gpu)
    d = torch.empty((B, 23), dtype=torch.int32, device=gpu)
    m = torch.empty(B, dtype=torch.int32, device=gpu)
    w4v_mod.ngram_draft(c, l, 1, 4, 23, out=d, match=m, ws=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4v_mod.ngram_draft(c, l, 1, 4, 23, out=d, match=m, ws=ws)
    for _ in range(3):
        d.fill_(-9)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(d.cpu().numpy(), d_o) and np.array_equal(m.cpu().numpy(), m_o)
    assert torch.all(ws == 0)


def test_drafts_feed_the_fused_verify(w4v_mod, gpu, oracle_mod):
    """Drafter -> verify on the device: n-gram drafts of 8 rows go straight
    into w8_lmhead_argmax_accept, whose acceptance equals the oracle's on the
    same target tokens."""
    B, nd, H, V = 8, 15, 256, 1024
    ctx, lens = inputs.ngram_contexts(5, B, 2048, V, "verify")
    d, _ = w4v_mod.ngram_draft(to_dev(ctx, gpu), to_dev(lens, gpu), 1, 4, nd)
    X = inputs.activations(5, B * (nd + 1), H, "ngram-verify")
    W, s = inputs.lmhead_weights(5, V, H, "ngram-verify")
    tok, n, out = w4v_mod.w8_lmhead_argmax_accept(to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu), d)
    torch.cuda.synchronize()
    d_o, _ = oracle_mod.ngram_draft(ctx, lens, 1, 4, nd)
    assert np.array_equal(d.cpu().numpy(), d_o)
    n_o, out_o = oracle_mod.spec_accept(tok.cpu().numpy().reshape(B, nd + 1), d_o)
    assert np.array_equal(n.cpu().numpy(), n_o) and np.array_equal(out.cpu().numpy(), out_o)
