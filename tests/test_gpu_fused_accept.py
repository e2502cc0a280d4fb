"""w8_lmhead_argmax_accept on the GPU: the lm_head argmax and the greedy
acceptance in one launch ("Efficient LLM Challenge Results", section 3: the
target checks all K+1 positions in one pass and keeps the longest draft
prefix equal to its own greedy tokens; -1 sentinels are never accepted).

Bit-exact against the oracle given identical logits: the fused tokens equal
the oracle's argmax over the kernel's own fp32 logits (read back through
w8_lmhead_argmax's testing-only output), and the accepted lengths and
emitted tokens equal the oracle's acceptance over those tokens.  The drafts
are drawn from the target tokens (the verify rows do not depend on them), so
every acceptance length occurs."""
import numpy as np
import pytest
import torch

from helpers import to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _plain_tokens(w4v_mod, gpu, X, W, s):
    M, V = X.shape[0], W.shape[0]
    logits = torch.empty((M, V), dtype=torch.float32, device=gpu)
    tok = w4v_mod.w8_lmhead_argmax(to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu), logits=logits)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), logits.cpu().numpy()


def _fused_vs_oracle(w4v_mod, gpu, oracle_mod, B, nd, K, V, seed, alpha=None, pad=False):
    M = B * (nd + 1)
    X = inputs.activations(seed, M, K, "fused-x")
    W, s = inputs.lmhead_weights(seed, V, K, "fused")
    t_plain, logits = _plain_tokens(w4v_mod, gpu, X, W, s)
    assert np.array_equal(t_plain, oracle_mod.argmax(logits))
    t = t_plain.reshape(B, nd + 1)
    if pad:
        d, _ = inputs.drafts_padded(seed, t, V, alpha, "fused")
    else:
        d = inputs.drafts_alpha(seed, t, V, alpha, "fused")
    d = np.ascontiguousarray(d.reshape(B, nd), dtype=np.int32)
    tok, n, out = w4v_mod.w8_lmhead_argmax_accept(to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu), to_dev(d, gpu))
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), t_plain)
    n_o, out_o = oracle_mod.spec_accept(t, d)
    assert np.array_equal(n.cpu().numpy(), n_o)
    assert np.array_equal(out.cpu().numpy(), out_o)
    assert w4v_mod.get_status() == 0
    return n_o


@pytest.mark.parametrize("B,nd,K,V,alpha,pad", [
    (1, 15, 256, 1024, 0.5, False),     # the tiny verify step's lm_head + acceptance
    (1, 15, 256, 1024, 1.0, False),     # all accepted: K+1 tokens out
    (1, 15, 256, 1024, 0.0, False),     # all rejected
    (1, 20, 384, 1000, 0.9, True),      # K = 20 padded with -1 sentinels
    (8, 15, 256, 2048, None, False),    # 8 verify blocks, acceptance rate set by the seed
    (4, 0, 128, 136, None, False),      # no drafts: n = 0, out = the target's token
    (2, 63, 128, 520, 0.97, False),     # 64 positions per block: two ballot rounds
    (128, 0, 128, 256, None, False),    # 128 blocks of one position
    (5, 24, 256, 1032, 0.8, True),      # 125 rows, blocks straddling 16-row MMA blocks
    (3, 1, 640, 3000, 1.0, False),
])
def test_fused_matches_oracle(w4v_mod, gpu, oracle_mod, B, nd, K, V, alpha, pad):
    n = _fused_vs_oracle(w4v_mod, gpu, oracle_mod, B, nd, K, V, seed=B * 100 + nd, alpha=alpha, pad=pad)
    if alpha == 1.0 and not pad:
        assert np.all(n == nd)
    if alpha == 0.0:
        assert np.all(n == 0)


def test_fused_full_vocab_batched(w4v_mod, gpu, oracle_mod):
    """Batched verify of 8 sequences x 16 positions (M = 128) through the
    2560 -> 151936 int8 lm_head, drafts with the per-seed acceptance rate."""
    _fused_vs_oracle(w4v_mod, gpu, oracle_mod, 8, 15, inputs.H_4B, inputs.V_4B, seed=4)


def test_fused_m16_full_vocab(w4v_mod, gpu, oracle_mod):
    """The verify step's own shape: one block of 15 drafts + 1."""
    _fused_vs_oracle(w4v_mod, gpu, oracle_mod, 1, 15, inputs.H_4B, inputs.V_4B, seed=1, alpha=0.75)


def test_fused_reuses_workspace_and_graphs(w4v_mod, gpu, oracle_mod):
    """Repeated calls on one workspace, captured in a CUDA graph and replayed,
    give the same tokens and lengths every time (the workspace is left zeroed)."""
    B, nd, K, V = 2, 15, 256, 4096
    X = inputs.activations(7, B * (nd + 1), K, "fused-g")
    W, s = inputs.lmhead_weights(7, V, K, "fused-g")
    t_plain, _ = _plain_tokens(w4v_mod, gpu, X, W, s)
    d = inputs.drafts_alpha(7, t_plain.reshape(B, nd + 1), V, 0.8, "g")
    Xd, Wd, sd, dd = to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu), to_dev(d, gpu)
    ws = w4v_mod.workspace(w4v_mod.w8_lmhead_argmax_workspace_bytes(B * (nd + 1), V), gpu)
    tok = torch.empty(B * (nd + 1), dtype=torch.int32, device=gpu)
    n = torch.empty(B, dtype=torch.int32, device=gpu)
    out = torch.empty((B, nd + 1), dtype=torch.int32, device=gpu)
    call = lambda: w4v_mod.w8_lmhead_argmax_accept(Xd, Wd, sd, dd, out=tok, n_out=n, tok_out=out, ws=ws)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    n_o, out_o = oracle_mod.spec_accept(t_plain.reshape(B, nd + 1), d)
    for _ in range(3):
        n.fill_(-7)
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), t_plain)
        assert np.array_equal(n.cpu().numpy(), n_o)
        assert np.array_equal(out.cpu().numpy(), out_o)
    assert torch.all(ws == 0)
    assert w4v_mod.get_status() == 0


@pytest.mark.parametrize("B,nd,V", [(8, 15, inputs.V_4B), (5, 24, 2048), (2, 63, 520)])
def test_fused_batch_invariant(w4v_mod, gpu, oracle_mod, B, nd, V):
    """W4V_BATCH_INVARIANT with more than 32 rows: the argmax in 32-row blocks,
    then the acceptance over every block.  Each sequence's tokens equal the
    tokens of that sequence's rows verified alone, and the accepted lengths
    and emitted tokens are the oracle's acceptance of them."""
    K = inputs.H_4B if V == inputs.V_4B else 256
    M = B * (nd + 1)
    X = inputs.activations(B + nd, M, K, "binv-x")
    W, s = inputs.lmhead_weights(B + nd, V, K, "binv")
    Xd, Wd, sd = to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu)
    alone = np.concatenate([w4v_mod.w8_lmhead_argmax(Xd[b * (nd + 1):(b + 1) * (nd + 1)].contiguous(), Wd, sd)
                            .cpu().numpy() for b in range(B)])
    t = alone.reshape(B, nd + 1)
    d = np.ascontiguousarray(inputs.drafts_alpha(B + nd, t, V, 0.8, "binv").reshape(B, nd), dtype=np.int32)
    tok, n, out = w4v_mod.w8_lmhead_argmax_accept(Xd, Wd, sd, to_dev(d, gpu), batch_invariant=True)
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), alone)
    n_o, out_o = oracle_mod.spec_accept(t, d)
    assert np.array_equal(n.cpu().numpy(), n_o)
    assert np.array_equal(out.cpu().numpy(), out_o)
    assert w4v_mod.get_status() == 0
