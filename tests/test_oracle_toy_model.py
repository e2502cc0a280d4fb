"""The invariant that pins the verify step end to end.

"Efficient LLM Challenge Results", section 3: under greedy verification
speculative decoding leaves the output unchanged, whatever the drafts; drafts
padded with -1 sentinels stay lossless.  On a toy W4A16 target with an int8
lm_head (oracle/toy_model.py), speculative decoding with random, perfect,
perfect-then-wrong, all-sentinel, prompt-lookup (n-gram), K=0, K=15, K=20
and K=23 drafters must emit the same tokens as plain greedy decoding, token
for token.
"""
import numpy as np
import pytest

import oracle
from oracle.toy_model import ToyWeights, greedy_decode, spec_decode
from speculative_decoding_verify_w4a16_gb300 import inputs


def _weights(seed, V):
    E, layers, W8, s8 = inputs.toy_model_arrays(seed, V=V, H=256, layers=2)
    return ToyWeights(E, layers, W8, s8)


def _drafters(w, seed):
    rng = np.random.default_rng(seed)
    V = w.V

    def random(ctx, K):
        return [int(x) for x in rng.integers(0, V, K)]

    def perfect(ctx, K):
        return greedy_decode(w, ctx, K)

    def perfect_then_wrong(ctx, K):
        good = greedy_decode(w, ctx, K)
        j = int(rng.integers(0, K + 1))
        tail = [(g + 1 + int(rng.integers(0, V - 1))) % V for g in good[j:]]
        return good[:j] + tail

    def sentinel(ctx, K):
        return [-1] * K

    def padded(ctx, K):
        L = int(rng.integers(0, K + 1))
        return greedy_decode(w, ctx, L) + [-1] * (K - L)

    def ngram(ctx, K):
        # prompt lookup over the context so far (the oracle's n-gram drafter)
        d, _ = oracle.ngram_draft(np.array(ctx, np.int32), None, 1, 3, K)
        return [int(x) for x in d]

    return dict(random=random, perfect=perfect, perfect_then_wrong=perfect_then_wrong,
                sentinel=sentinel, padded=padded, ngram=ngram)


CASES = (("random", 15), ("perfect", 15), ("perfect_then_wrong", 15),
         ("sentinel", 20), ("padded", 20), ("random", 0), ("perfect", 4), ("ngram", 15), ("ngram", 23))


@pytest.mark.parametrize("V", [64, 1024])
def test_spec_decode_equals_greedy(V):
    w = _weights(11, V)
    n_prompts = 6 if V == 64 else 3
    n_new = 24
    for p in range(n_prompts):
        prompt = inputs.random_tokens(100 + p, 1 + p % 5, V)
        want = greedy_decode(w, prompt, n_new)
        drafters = _drafters(w, 1000 + p)
        for name, K in CASES:
            stats = {}
            got = spec_decode(w, prompt, n_new, K, drafters[name], stats)
            assert got == want, (V, p, name, K)
            if name == "perfect" and K > 0:
                # a perfect drafter is fully accepted: K+1 tokens per verify step
                assert stats["steps"] == -(-n_new // (K + 1))
            if name == "sentinel":
                assert stats["accepted"] == 0


@pytest.mark.slow
def test_spec_decode_equals_greedy_many_prompts():
    w = _weights(12, 64)
    for p in range(100):
        prompt = inputs.random_tokens(500 + p, 1 + p % 7, 64)
        want = greedy_decode(w, prompt, 20)
        drafters = _drafters(w, 2000 + p)
        for name, K in (("random", 15), ("perfect_then_wrong", 15), ("padded", 20)):
            assert spec_decode(w, prompt, 20, K, drafters[name]) == want, (p, name)


def test_toy_model_is_context_dependent():
    """Guards the invariant test against a degenerate model whose greedy output
    ignores the context (which would make it pass trivially)."""
    w = _weights(11, 64)
    outs = {tuple(greedy_decode(w, inputs.random_tokens(300 + i, 3, 64), 12)) for i in range(8)}
    assert len(outs) >= 4
    seq = greedy_decode(w, [1, 2, 3], 24)
    assert len(set(seq)) >= 3


# ------------------------------------------------- recurrent (gated-delta) state
def _weights_gdn(seed, V):
    E, layers, W8, s8 = inputs.toy_model_arrays(seed, V=V, H=256, layers=2)
    return ToyWeights(E, layers, W8, s8, gdn=inputs.toy_gdn_arrays(seed, H=256, heads=2))


GDN_CASES = (("random", 15), ("perfect_then_wrong", 15), ("padded", 20), ("sentinel", 20),
             ("ngram", 15), ("perfect", 4), ("random", 0))


def test_spec_decode_equals_greedy_with_recurrent_state():
    """With a gated-delta layer, speculative decoding commits only the accepted
    prefix of each verify block and still emits exactly the greedy tokens
    (greedy recomputes the state from the first token at every step)."""
    w = _weights_gdn(21, 64)
    n_new = 16
    for p in range(3):
        prompt = inputs.random_tokens(300 + p, 2 + p, 64)
        want = greedy_decode(w, prompt, n_new)
        drafters = _drafters(w, 3000 + p)
        for name, K in GDN_CASES:
            stats = {}
            got = spec_decode(w, prompt, n_new, K, drafters[name], stats)
            assert got == want, (p, name, K)
            if name == "perfect":
                assert stats["steps"] == -(-n_new // (K + 1))


def test_invariant_catches_a_corrupted_recurrent_state():
    """The two failures the pages describe, planted in the oracle on the CPU:
    committing the rejected positions' updates, or never advancing the state
    (a stale state), each change the emitted tokens for some prompt."""
    w = _weights_gdn(22, 64)
    n_new = 16
    caught = {"all": False, "none": False}
    for p in range(4):
        prompt = inputs.random_tokens(400 + p, 3, 64)
        want = greedy_decode(w, prompt, n_new)
        for mode in caught:
            rng = np.random.default_rng(4000 + p)
            drafter = lambda ctx, K: [int(x) for x in rng.integers(0, 64, K)]
            if spec_decode(w, prompt, n_new, 15, drafter, commit=mode) != want:
                caught[mode] = True
        if all(caught.values()):
            break
    assert caught == {"all": True, "none": True}


def test_recurrent_state_matters():
    """The layer's state changes the tokens: the same context with the state
    reset to zero before the last position gives different logits."""
    from oracle.toy_model import logits_at
    w = _weights_gdn(23, 64)
    toks = inputs.random_tokens(500, 12, 64)
    L1 = logits_at(w, toks, [11])
    L0 = logits_at(w, toks, [11], state=w.zero_state())
    assert not np.allclose(L1, L0)
