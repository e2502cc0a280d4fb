"""Speculative decoding through the library's kernels emits exactly the greedy
tokens ("Efficient LLM Challenge Results", section 3: greedy verification
leaves the output unchanged whatever the drafts; padded -1 drafts stay
lossless; "DFlash K=15 for Qwen3.5-4B on a single A10G", "What transfers":
a rejected draft must not corrupt a recurrent state).

The toy target of oracle/toy_model.py (gated-delta layer, two W4A16 MLP
layers, int8 lm_head) runs with every projection, the recurrent state, the
lm_head argmax and the acceptance on the GPU (w4a16_gemm, gdn_verify /
gdn_commit, w8_lmhead_argmax, spec_accept, ngram_draft); only the
position-wise glue (embedding, rms, silu, gates) is numpy on the host.
Greedy decoding runs one position per step through the same kernels.  Exact
equality needs every kernel to give a row the same result whatever the
number of rows beside it (M = 1 against M = K+1) and the committed state to
be exactly the one-position-at-a-time state: the verify-sized GEMM and the
lm_head are built batch-invariant for M <= 32, and the recurrence runs the
same fp32 steps in both cases.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu

H, V, HEADS, D = 256, 1024, 2, 128
RMS_EPS = 1e-6


def _rms(x):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + RMS_EPS)


class GpuToy:
    def __init__(self, w4v, gpu, seed):
        self.w4v, self.gpu = w4v, gpu
        E, layers, W8, s8 = inputs.toy_model_arrays(seed, V=V, H=H, layers=2)
        q_qkv, s_qkv, q_o, s_o, wa, wb = inputs.toy_gdn_arrays(seed, H=H, heads=HEADS)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(gpu)
        pk = lambda q: dev(w4v.pack_int4(q))
        self.E = E.astype(np.float64)
        self.qkv = (pk(q_qkv), dev(s_qkv), q_qkv.shape[0])
        self.o = (pk(q_o), dev(s_o), q_o.shape[0])
        self.wa, self.wb = wa.astype(np.float64), wb.astype(np.float64)
        self.layers = [((pk(a), dev(b), a.shape[0]), (pk(c), dev(d), c.shape[0])) for (a, b, c, d) in layers]
        self.W8, self.s8 = dev(W8), dev(s8)

    def gemm(self, x16, w):
        # more than 32 rows (several sequences' verify blocks) in 32-row blocks,
        # so that every row is computed as it would be alone
        packed, s, N = w
        out = self.w4v.w4a16_gemm(torch.from_numpy(np.ascontiguousarray(x16)).to(self.gpu), packed, s, N,
                                  batch_invariant=True)
        return out.cpu().numpy().astype(np.float64)

    def inputs_at(self, tokens, p0, T):
        emb = self.E[np.asarray(tokens, np.int64)]
        csum = np.cumsum(emb, axis=0)
        pos = np.arange(p0, p0 + T)
        return emb[pos] + csum[pos] / (pos[:, None] + 1.0)

    def gdn_inputs(self, h, B=1):
        """The recurrence's inputs for B sequences' blocks of T positions each
        (h holds the B*T rows one block after the other)."""
        T = h.shape[0] // B
        r = _rms(h).astype(np.float16)
        qkv = self.gemm(r, self.qkv)
        q = qkv[:, :H].reshape(B * T, HEADS, D)
        k = qkv[:, H:2 * H].reshape(B * T, HEADS, D)
        v = qkv[:, 2 * H:].reshape(B * T, HEADS, D)
        q = q / np.linalg.norm(q, axis=-1, keepdims=True)
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
        rd = r.astype(np.float64)
        alpha = 1.0 / (1.0 + np.exp(-(2.0 + rd @ self.wa.T)))
        beta = 1.0 / (1.0 + np.exp(-(rd @ self.wb.T)))
        dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a.reshape(B, T, *a.shape[1:]).astype(dt))).to(
            self.gpu)
        return (dev(q, np.float16), dev(k, np.float16), dev(v, np.float16),
                dev(alpha, np.float32), dev(beta, np.float32))

    def tokens_at(self, tokens, p0, T, S, pending=None):
        """Greedy tokens after positions p0..p0+T-1 from committed state S (not
        written); returns (tokens, the recurrence's inputs for a later commit).
        With `pending` = (inputs, n) of the previous block, that block's commit
        runs first, in the same launch (gdn_step)."""
        h = self.inputs_at(tokens, p0, T)
        q, k, v, a, b = self.gdn_inputs(h)
        if pending is None:
            o = self.w4v.gdn_verify(S, q, k, v, a, b)
        else:
            (kp, vp, ap, bp), n = pending
            nt = torch.tensor([n], dtype=torch.int32, device=self.gpu)
            o = self.w4v.gdn_step(S, (kp, vp, ap, bp, nt), q, k, v, a, b)
        h = h + self.gemm(o.cpu().numpy().reshape(T, H), self.o)
        for (w_gu, w_d) in self.layers:
            gu = self.gemm(_rms(h).astype(np.float16), w_gu)
            act = (gu[:, :H] / (1.0 + np.exp(-gu[:, :H]))) * gu[:, H:]
            h = h + self.gemm(act.astype(np.float16), w_d)
        X = torch.from_numpy(_rms(h).astype(np.float16)).to(self.gpu)
        t = self.w4v.w8_lmhead_argmax(X, self.W8, self.s8).cpu().numpy()
        return t, (k, v, a, b)

    def commit(self, S, gdn_in, n):
        k, v, a, b = gdn_in
        self.w4v.gdn_commit(S, k, v, a, b, torch.tensor([n], dtype=torch.int32, device=self.gpu))

    def fresh_state(self, tokens):
        S = torch.zeros((1, HEADS, D, D), dtype=torch.float32, device=self.gpu)
        L = len(tokens)
        if L > 1:
            _, gin = self.tokens_at(tokens, 0, L - 1, S)
            self.commit(S, gin, L - 2)
        return S

    def greedy(self, prompt, n_new):
        ctx = list(prompt)
        S = self.fresh_state(ctx)
        out = []
        while len(out) < n_new:
            t, gin = self.tokens_at(ctx, len(ctx) - 1, 1, S)
            self.commit(S, gin, 0)
            ctx.append(int(t[0]))
            out.append(int(t[0]))
        return out

    def spec(self, prompt, n_new, K, drafter, fused=False):
        ctx = list(prompt)
        S = self.fresh_state(ctx)
        out, steps = [], 0
        pending = None
        while len(out) < n_new:
            d = np.asarray(drafter(ctx, K), np.int32).reshape(1, K)
            seq = ctx + [int(x) if x >= 0 else 0 for x in d[0]]
            t, gin = self.tokens_at(seq, len(ctx) - 1, K + 1, S, pending)
            n, tok = self.w4v.spec_accept(torch.from_numpy(t.reshape(1, K + 1)).to(self.gpu),
                                          torch.from_numpy(d).to(self.gpu))
            n = int(n.cpu()[0])
            if fused:
                pending = (gin, n)                 # committed by the next block's launch
            else:
                self.commit(S, gin, n)             # only positions 0..n of the block
            emitted = [int(x) for x in tok.cpu().numpy()[0, : n + 1]]
            ctx.extend(emitted)
            out.extend(emitted)
            steps += 1
        return out[:n_new], steps


@pytest.mark.parametrize("seed", [31, 32])
def test_spec_equals_greedy_through_the_kernels(w4v_mod, gpu, seed):
    toy = GpuToy(w4v_mod, gpu, seed)
    prompt = inputs.random_tokens(600 + seed, 4, V)
    n_new = 24
    want = toy.greedy(prompt, n_new)
    rng = np.random.default_rng(seed)

    def random_drafts(ctx, K):
        return [int(x) for x in rng.integers(0, V, K)]

    def oracle_perfect(ctx, K):
        # the greedy continuation, known from the reference run; wrong after a seeded cut
        done = len(ctx) - len(prompt)
        good = (want + [0] * (K + 1))[done:done + K]
        cut = int(rng.integers(0, K + 1))
        return good[:cut] + [(g + 1) % V for g in good[cut:]]

    def padded(ctx, K):
        done = len(ctx) - len(prompt)
        L = int(rng.integers(0, K + 1))
        return (want + [0] * (K + 1))[done:done + L] + [-1] * (K - L)

    def ngram(ctx, K):
        c = torch.tensor([ctx], dtype=torch.int32, device=gpu)
        d, _ = w4v_mod.ngram_draft(c, torch.tensor([len(ctx)], dtype=torch.int32, device=gpu), 1, 3, K)
        return [int(x) for x in d.cpu().numpy()[0]]

    for name, drafter, K in (("random", random_drafts, 15), ("perfect_then_wrong", oracle_perfect, 15),
                             ("padded", padded, 20), ("ngram", ngram, 15)):
        got, steps = toy.spec(prompt, n_new, K, drafter)
        assert got == want, (seed, name)
        if name == "perfect_then_wrong":
            assert steps < n_new                    # accepted drafts did advance several tokens a step
    # the previous block's commit fused into the next block's launch (gdn_step)
    got, _ = toy.spec(prompt, n_new, 15, oracle_perfect, fused=True)
    assert got == want, (seed, "fused commit")
    assert w4v_mod.get_status() == 0


def test_commit_all_corrupts_the_recurrent_state(w4v_mod, gpu):
    """Committing the whole block (the rejected positions too) instead of the
    accepted prefix changes the emitted tokens: the invariant above is not
    satisfied by accident."""
    toy = GpuToy(w4v_mod, gpu, 33)
    prompt = inputs.random_tokens(700, 4, V)
    want = toy.greedy(prompt, 24)
    rng = np.random.default_rng(5)
    orig_commit = toy.commit
    toy.commit = lambda S, gin, n: orig_commit(S, gin, 15)   # planted: always all K+1 positions
    got, _ = toy.spec(prompt, 24, 15, lambda ctx, K: [int(x) for x in rng.integers(0, V, K)])
    assert got != want


def spec_batched(toy, prompts, n_new, K, drafter):
    """Speculative decoding of several sequences at once: one verify pass over
    every sequence's block of K+1 positions (B*(K+1) rows in each GEMM, the
    recurrent state of all B sequences, the lm_head argmax with each
    sequence's acceptance in one call), all in batch-invariant mode."""
    w4v, gpu = toy.w4v, toy.gpu
    B, T = len(prompts), K + 1
    ctxs = [list(p) for p in prompts]
    S = torch.cat([toy.fresh_state(c) for c in ctxs], dim=0)
    outs = [[] for _ in range(B)]
    while min(len(o) for o in outs) < n_new:
        d = np.stack([np.asarray(drafter(b, ctxs[b], K), np.int32) for b in range(B)])
        h = np.concatenate([toy.inputs_at(ctxs[b] + [int(x) if x >= 0 else 0 for x in d[b]], len(ctxs[b]) - 1, T)
                            for b in range(B)])
        q, k, v, a, be = toy.gdn_inputs(h, B)
        o = w4v.gdn_verify(S, q, k, v, a, be)
        h = h + toy.gemm(o.cpu().numpy().reshape(B * T, H), toy.o)
        for (w_gu, w_d) in toy.layers:
            gu = toy.gemm(_rms(h).astype(np.float16), w_gu)
            act = (gu[:, :H] / (1.0 + np.exp(-gu[:, :H]))) * gu[:, H:]
            h = h + toy.gemm(act.astype(np.float16), w_d)
        X = torch.from_numpy(_rms(h).astype(np.float16)).to(gpu)
        _, n, tok = w4v.w8_lmhead_argmax_accept(X, toy.W8, toy.s8, torch.from_numpy(d).to(gpu),
                                                batch_invariant=True)
        w4v.gdn_commit(S, k, v, a, be, n)              # each sequence keeps positions 0..n[b]
        n, tok = n.cpu().numpy(), tok.cpu().numpy()
        for b in range(B):
            emitted = [int(x) for x in tok[b, : n[b] + 1]]
            ctxs[b].extend(emitted)
            outs[b].extend(emitted)
    return [o[:n_new] for o in outs]


def test_batched_spec_equals_greedy_through_the_kernels(w4v_mod, gpu):
    """8 sequences verified together, 16 positions each (128 rows per GEMM and
    in the lm_head, one recurrent state per sequence): every sequence emits
    exactly its own one-position greedy tokens, for random drafts and for
    drafts that follow the greedy continuation up to a seeded cut."""
    toy = GpuToy(w4v_mod, gpu, 34)
    B, n_new, K = 8, 20, 15
    prompts = [inputs.random_tokens(800 + b, 4, V) for b in range(B)]
    want = [toy.greedy(p, n_new) for p in prompts]
    rng = np.random.default_rng(34)

    def random_drafts(b, ctx, K):
        return [int(x) for x in rng.integers(0, V, K)]

    def perfect_then_wrong(b, ctx, K):
        # (a sequence already past n_new tokens, waiting for the others, gets zeros)
        done = len(ctx) - len(prompts[b])
        good = (want[b] + [0] * (done + K + 1))[done:done + K]
        cut = int(rng.integers(0, K + 1))
        return good[:cut] + [(g + 1) % V for g in good[cut:]]

    for name, drafter in (("random", random_drafts), ("perfect_then_wrong", perfect_then_wrong)):
        got = spec_batched(toy, prompts, n_new, K, drafter)
        for b in range(B):
            assert got[b] == want[b], (name, b)
    assert w4v_mod.get_status() == 0
