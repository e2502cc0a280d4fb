"""w8_lmhead_argmax on the GPU against the oracle.

The greedy token must be bit-exact given identical logits: the fused
kernel's token equals the oracle's argmax over the kernel's own fp32 logits
(read back through the testing-only logits output).  Against the oracle's
double-precision logits every logit is within the fp32 summation bound, and
a token can differ from the oracle's only where the two best logits are
closer than that bound.
"""
import numpy as np
import pytest
import torch

from helpers import logit_bound, to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _run(w4v_mod, gpu, X, W, s, debug=True, batch_invariant=False):
    M = X.shape[0]
    V = W.shape[0]
    Xd, Wd, sd = to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu)
    maxl = torch.empty(M, dtype=torch.float32, device=gpu)
    logits = torch.empty((M, V), dtype=torch.float32, device=gpu) if debug else None
    tok = w4v_mod.w8_lmhead_argmax(Xd, Wd, sd, maxlogit=maxl, logits=logits, batch_invariant=batch_invariant)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), maxl.cpu().numpy(), (logits.cpu().numpy() if debug else None)


def _check(oracle_mod, X, W, s, tok, maxl, logits):
    M = X.shape[0]
    # bit-exact given identical logits
    assert np.array_equal(tok, oracle_mod.argmax(logits))
    assert np.array_equal(maxl, logits[np.arange(M), tok])
    # the kernel's logits against the definition, within the fp32 bound
    L = oracle_mod.lmhead_logits(X, W, s)
    bound = logit_bound(X, W, s)
    assert np.all(np.abs(logits - L) <= bound)
    # token against the oracle's own token: equal unless a near-tie
    t_o = oracle_mod.argmax(L)
    for m in np.nonzero(tok != t_o)[0]:
        gap = L[m, t_o[m]] - L[m, tok[m]]
        assert gap <= bound[m, t_o[m]] + bound[m, tok[m]], (m, gap)
    return int(np.sum(tok != t_o))


def test_cfg0_lmhead(w4v_mod, gpu, oracle_mod):
    """Tiny verify step: 16 rows through a 256 -> 1024 int8 lm_head."""
    X = inputs.activations(0, 16, 256, "cfg0-x")
    W, s = inputs.lmhead_weights(0, 1024, 256, "cfg0")
    tok, maxl, logits = _run(w4v_mod, gpu, X, W, s)
    assert _check(oracle_mod, X, W, s, tok, maxl, logits) == 0


@pytest.mark.parametrize("M,K,V", [(1, 256, 1024), (3, 128, 136), (16, 384, 1000), (21, 256, 2048),
                                   (32, 512, 1032), (48, 1280, 296), (64, 256, 520), (100, 128, 4096),
                                   (128, 640, 3000), (128, 256, 38408)])
def test_shapes(w4v_mod, gpu, oracle_mod, M, K, V):
    X = inputs.activations(M, M, K, "x")
    W, s = inputs.lmhead_weights(V, V, K)
    tok, maxl, logits = _run(w4v_mod, gpu, X, W, s)
    assert _check(oracle_mod, X, W, s, tok, maxl, logits) == 0


def test_ties_go_to_lowest_index(w4v_mod, gpu, oracle_mod):
    """Identical vocabulary rows in different tiles give bit-identical logits;
    the lowest index must win."""
    M, K, V = 8, 256, 1024
    X = inputs.activations(5, M, K, "tie")
    W, s = inputs.lmhead_weights(5, V, K, "tie")
    s = s.copy()
    W = W.copy()
    for v in (37, 300, 900):
        W[v] = W[700]
        s[v] = np.float16(0.5)
    s[700] = np.float16(0.5)
    X = X.copy()
    dot = X.astype(np.float64) @ W[700].astype(np.float64)
    X[dot < 0] = -X[dot < 0]                     # make the tied rows' logits positive and large
    tok, maxl, logits = _run(w4v_mod, gpu, X, W, s)
    assert np.all(tok == 37)
    assert np.all(logits[:, 37] == logits[:, 900])
    _check(oracle_mod, X, W, s, tok, maxl, logits)


def test_constant_and_nan_rows(w4v_mod, gpu, oracle_mod):
    M, K, V = 4, 128, 512
    X = np.zeros((M, K), np.float16)
    X[1, :] = 1.0
    X[2, 5] = np.float16("nan")
    W, s = inputs.lmhead_weights(9, V, K)
    W = W.copy()
    W[:, :] = 3                                   # every logit of a row equal (or all NaN)
    s = np.full(V, 0.25, np.float16)
    tok, maxl, logits = _run(w4v_mod, gpu, X, W, s)
    assert list(tok) == [0, 0, 0, 0]
    assert np.array_equal(tok, oracle_mod.argmax(logits))


def test_workspace_reuse_is_clean(w4v_mod, gpu):
    M, K, V = 16, 256, 2048
    X = to_dev(inputs.activations(1, M, K), gpu)
    W, s = inputs.lmhead_weights(1, V, K)
    Wd, sd = to_dev(W, gpu), to_dev(s, gpu)
    ws = w4v_mod.workspace(w4v_mod.w8_lmhead_argmax_workspace_bytes(M, V), gpu)
    a = w4v_mod.w8_lmhead_argmax(X, Wd, sd, ws=ws).cpu().numpy()
    b = w4v_mod.w8_lmhead_argmax(X, Wd, sd, ws=ws).cpu().numpy()
    assert np.array_equal(a, b)
    assert np.all(ws.cpu().numpy() == 0)      # keys and counter left cleared
    assert w4v_mod.get_status() == 0


def test_full_vocab_cfg1(w4v_mod, gpu, oracle_mod):
    """The 4B-shaped lm_head (2560 -> 151936) at M = 16."""
    M, K, V = 16, 2560, 151936
    X = inputs.activations(1, M, K, "cfg1-lm")
    W, s = inputs.lmhead_weights(1, V, K, "cfg1")
    tok, maxl, logits = _run(w4v_mod, gpu, X, W, s)
    assert np.array_equal(tok, oracle_mod.argmax(logits))
    r = np.random.default_rng(0)
    vs = np.sort(r.choice(V, 3000, replace=False))
    vs = np.unique(np.concatenate([vs, tok]))
    L = oracle_mod.lmhead_logits(X, W[vs], s[vs])
    bound = logit_bound(X, W[vs], s[vs])
    assert np.all(np.abs(logits[:, vs] - L) <= bound)
    t_o, best, second = oracle_mod.lmhead_argmax_rows(X, W, s, np.arange(M, dtype=np.int32))
    for m in range(M):
        if tok[m] != t_o[m]:
            # the kernel may only prefer another token where the fp32 error
            # bounds of the two logits overlap: L(t_o) - L(tok) <= b(t_o) + b(tok)
            pair = np.array([t_o[m], tok[m]])
            Lp = oracle_mod.lmhead_logits(X[m:m + 1], W[pair], s[pair])[0]
            bp = logit_bound(X[m:m + 1], W[pair], s[pair])[0]
            assert Lp[0] - Lp[1] <= bp[0] + bp[1], m


def test_batch_invariance(w4v_mod, gpu):
    """For M <= 32 every logit comes from the same arithmetic whatever M is:
    the rows of a small call equal the same rows of a 32-row call bit for
    bit (logits and tokens)."""
    K, V = 512, 4096
    X = inputs.activations(77, 32, K, "inv")
    W, s = inputs.lmhead_weights(77, V, K, "inv")
    tok32, _, L32 = _run(w4v_mod, gpu, X, W, s)
    for m in (1, 7, 16, 17, 21):
        tok, _, L = _run(w4v_mod, gpu, X[:m], W, s)
        assert np.array_equal(L, L32[:m]), m
        assert np.array_equal(tok, tok32[:m]), m


def test_batch_invariance_batched_verify(w4v_mod, gpu, oracle_mod):
    """With W4V_BATCH_INVARIANT the batched verify of 8 sequences x 16
    positions (128 rows in one call) gives every row the logits and token of
    the same row verified alone (16 rows) and decoded alone (1 row), bit for
    bit, so batching never changes an accepted token.  Without the flag the
    128 rows run in one launch that sums each logit in another order: every
    logit still within the fp32 bound of the oracle."""
    K, V = 2560, 8192
    X = inputs.activations(78, 128, K, "inv128")
    W, s = inputs.lmhead_weights(78, V, K, "inv128")
    _, _, Lfast = _run(w4v_mod, gpu, X, W, s)
    r = np.random.default_rng(78)
    vs = np.sort(r.choice(V, 600, replace=False))
    assert np.all(np.abs(Lfast[:, vs] - oracle_mod.lmhead_logits(X, W[vs], s[vs])) <= logit_bound(X, W[vs], s[vs]))
    tok128, _, L128 = _run(w4v_mod, gpu, X, W, s, batch_invariant=True)
    for b in range(8):
        tok, _, L = _run(w4v_mod, gpu, X[16 * b:16 * b + 16], W, s)
        assert np.array_equal(L, L128[16 * b:16 * b + 16]), b
        assert np.array_equal(tok, tok128[16 * b:16 * b + 16]), b
    for m in (0, 37, 127):
        tok, _, L = _run(w4v_mod, gpu, X[m:m + 1], W, s)
        assert np.array_equal(L[0], L128[m]), m
        assert tok[0] == tok128[m], m
