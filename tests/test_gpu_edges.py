"""Edge cases of the verify path on the GPU against the oracle: the smallest
legal shapes (one 8-row tile, one group, one vocabulary block), the largest
verify size and the first prefill size on either side of the kernel switch,
M = 0 no-ops that must leave outputs untouched, and one whole verify step
(W4A16 linear -> int8 lm_head argmax -> greedy acceptance) composed on the
device and checked end to end."""
import numpy as np
import pytest
import torch

from helpers import GEMM_TOL, gemm_rel_err, to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _gemm(w4v_mod, gpu, A, q, s, **kw):
    packed = to_dev(w4v_mod.pack_int4(q), gpu)
    C = w4v_mod.w4a16_gemm(to_dev(A, gpu), packed, to_dev(s, gpu), q.shape[0], **kw)
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (16, 8, 128), (32, 8, 128), (32, 8, 256), (33, 8, 128),
                                   (32, 136, 384), (33, 136, 384), (1, 2560, 128), (16, 8, 9728)])
def test_gemm_extreme_shapes(w4v_mod, gpu, oracle_mod, M, N, K):
    """One partial 8-row tile, one quantization group, the largest verify M
    (32) and the smallest prefill M (33), long K with a single tile."""
    A = inputs.activations(11, M, K, "edge")
    q = inputs.w4_codes(11, N, K, "edge")
    s = inputs.w4_scales(11, N, K, "edge")
    C = _gemm(w4v_mod, gpu, A, q, s)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s)) <= GEMM_TOL
    if M <= 32:
        C2 = _gemm(w4v_mod, gpu, A, q, s, static_weights=True)
        assert np.array_equal(C, C2)


def test_gemm_m0_is_a_noop(w4v_mod, gpu):
    N, K = 256, 256
    q = inputs.w4_codes(12, N, K, "noop")
    s = to_dev(inputs.w4_scales(12, N, K, "noop"), gpu)
    packed = to_dev(w4v_mod.pack_int4(q), gpu)
    A = torch.empty((0, K), dtype=torch.float16, device=gpu)
    out = torch.full((1, N), 7.0, dtype=torch.float16, device=gpu)
    w4v_mod.w4a16_gemm(A, packed, s, N, out=out[:0])
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


@pytest.mark.parametrize("M,K,V", [(1, 128, 8), (128, 128, 8), (128, 128, 136), (1, 128, 151936)])
def test_lmhead_extreme_shapes(w4v_mod, gpu, oracle_mod, M, K, V):
    """Smallest vocabulary (one partial 128-row block), the largest M (128),
    and the full vocabulary with one row (the prefill's last row)."""
    X = inputs.activations(13, M, K, "edge-x")
    W, s = inputs.lmhead_weights(13, V, K, "edge")
    logits = torch.empty((M, V), dtype=torch.float32, device=gpu)
    tok = w4v_mod.w8_lmhead_argmax(to_dev(X, gpu), to_dev(W, gpu), to_dev(s, gpu), logits=logits)
    torch.cuda.synchronize()
    tok, logits = tok.cpu().numpy(), logits.cpu().numpy()
    assert np.all((tok >= 0) & (tok < V))
    assert np.array_equal(tok, oracle_mod.argmax(logits))
    assert w4v_mod.get_status() == 0


def test_lmhead_m0_is_a_noop(w4v_mod, gpu):
    K, V = 128, 1024
    W, s = inputs.lmhead_weights(14, V, K, "noop")
    X = torch.empty((0, K), dtype=torch.float16, device=gpu)
    out = torch.full((4,), 123, dtype=torch.int32, device=gpu)
    w4v_mod.w8_lmhead_argmax(X, to_dev(W, gpu), to_dev(s, gpu), out=out[:0])
    torch.cuda.synchronize()
    assert torch.all(out == 123)


def test_composed_verify_step_cfg0(w4v_mod, gpu, oracle_mod):
    """The small configuration as one device step: a 256 -> 512 W4A16 linear
    (K = 15 drafts + 1 rows), a 512 -> 1024 int8 lm_head argmax on its
    output, then acceptance of 15 drafts with half forced to match; every
    stage on the GPU, compared with the oracle run on the GPU's own
    intermediate (so the comparison isolates each stage's rounding)."""
    M, H, I, V, Kd = 16, 256, 512, 1024, 15
    A = inputs.activations(0, M, H, "cfg0-a")
    q = inputs.w4_codes(0, I, H, "cfg0")
    s = inputs.w4_scales(0, I, H, "cfg0")
    W8, s8 = inputs.lmhead_weights(0, V, I, "cfg0-step")
    packed = to_dev(w4v_mod.pack_int4(q), gpu)
    h = w4v_mod.w4a16_gemm(to_dev(A, gpu), packed, to_dev(s, gpu), I, static_weights=True)
    logits = torch.empty((M, V), dtype=torch.float32, device=gpu)
    tok = w4v_mod.w8_lmhead_argmax(h, to_dev(W8, gpu), to_dev(s8, gpu), logits=logits)
    t = tok.reshape(1, M)
    d_host = inputs.drafts_half_match(0, t.cpu().numpy()[0], V).reshape(1, Kd)
    n, out = w4v_mod.spec_accept(t, to_dev(d_host, gpu))
    torch.cuda.synchronize()
    h_host = h.cpu().numpy()
    assert gemm_rel_err(h_host.astype(np.float64), oracle_mod.w4a16_gemm(A, q, s)) <= GEMM_TOL
    assert np.array_equal(tok.cpu().numpy(), oracle_mod.argmax(logits.cpu().numpy()))
    n_o, out_o = oracle_mod.spec_accept(t.cpu().numpy(), d_host)
    assert np.array_equal(n.cpu().numpy(), n_o)
    assert np.array_equal(out.cpu().numpy(), out_o)
    assert w4v_mod.get_status() == 0
