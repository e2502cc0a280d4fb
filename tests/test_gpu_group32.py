"""w4a16_gemm with group size 32 on the GPU against the oracle.

"Efficient LLM Challenge Results", section 5, lists a W4A16 target in the
compressed-tensors format with group size 32 beside the GPTQ group-128 one:
the same int4 codes and packed layout, one fp16 scale (and zero point) per 32
k instead of per 128.  Both kernels fold each sub-group's scale into the
dequantized fp16 weight; the bound is the same 2e-3 relative error, and the
per-element arithmetic of the verify-sized kernel still does not depend on M.
"""
import numpy as np
import pytest
import torch

from helpers import GEMM_TOL, gemm_rel_err, to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu
G = 32


def _gemm(w4v_mod, gpu, A, q, s, zeros=None, static_weights=False):
    packed = to_dev(w4v_mod.pack_int4(q), gpu)
    C = w4v_mod.w4a16_gemm(to_dev(A, gpu), packed, to_dev(s, gpu), q.shape[0],
                           zeros=None if zeros is None else to_dev(zeros, gpu),
                           static_weights=static_weights, group=G)
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64)


def _case(seed, M, N, K, zeros, tag):
    A = inputs.activations(seed, M, K, tag)
    q = inputs.w4_codes(seed, N, K, tag)
    s = inputs.w4_scales(seed, N, K, tag, group=G)
    z = inputs.w4_zeros(seed, N, K, tag, group=G) if zeros else None
    return A, q, s, z


@pytest.mark.parametrize("M,N,K", [(1, 512, 256), (16, 2560, 2560), (5, 200, 384), (21, 768, 1280),
                                   (32, 384, 2560), (16, 2560, 9728), (9, 384, 768), (31, 264, 1152),
                                   (16, 19456, 2560)])
def test_verify_sizes(w4v_mod, gpu, oracle_mod, M, N, K):
    A, q, s, _ = _case(M, M, N, K, False, "g32")
    C = _gemm(w4v_mod, gpu, A, q, s)
    if N * K <= 2560 * 9728:
        assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s, group=G)) <= GEMM_TOL
    else:
        r = np.random.default_rng(K)
        rows = r.integers(0, M, 4000).astype(np.int32)
        cols = r.integers(0, N, 4000).astype(np.int32)
        R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols, group=G)
        assert gemm_rel_err(C[rows, cols], R) <= GEMM_TOL


@pytest.mark.parametrize("M,N,K", [(16, 512, 512), (3, 272, 640), (24, 400, 3200), (96, 256, 512),
                                   (300, 272, 1280)])
def test_zero_points(w4v_mod, gpu, oracle_mod, M, N, K):
    """A zero point per (32-k sub-group, row), verify and prefill sizes."""
    A, q, s, z = _case(3, M, N, K, True, "g32z")
    C = _gemm(w4v_mod, gpu, A, q, s, zeros=z)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s, zeros=z, group=G)) <= GEMM_TOL


@pytest.mark.parametrize("M", [16, 21])
def test_zero_points_stream_k(w4v_mod, gpu, oracle_mod, M):
    """The gate_up shape (19456 x 2560, the stream-K split, where a CTA's
    range starts and ends inside tiles) with a group-32 zero table: sampled
    outputs and two full rows against the oracle."""
    N, K = 19456, 2560
    A, q, s, z = _case(13, M, N, K, True, "g32zk")
    C = _gemm(w4v_mod, gpu, A, q, s, zeros=z)
    r = np.random.default_rng(M + 32)
    rows = r.integers(0, M, 4000).astype(np.int32)
    cols = r.integers(0, N, 4000).astype(np.int32)
    rows = np.concatenate([rows, np.zeros(N, np.int32), np.full(N, M - 1, np.int32)])
    cols = np.concatenate([cols, np.arange(N, dtype=np.int32), np.arange(N, dtype=np.int32)])
    R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols, zeros=z, group=G)
    assert gemm_rel_err(C[rows, cols], R) <= GEMM_TOL


@pytest.mark.parametrize("M,N,K", [(33, 512, 256), (128, 2560, 2560), (200, 520, 640), (300, 384, 9728),
                                   (700, 2560, 512), (2048, 2560, 512)])
def test_prefill_sizes(w4v_mod, gpu, oracle_mod, M, N, K):
    A, q, s, _ = _case(M, M, N, K, False, "g32p")
    C = _gemm(w4v_mod, gpu, A, q, s)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s, group=G)) <= GEMM_TOL


@pytest.mark.parametrize("M", [16, 64])
def test_sub_group_scale_orientation(w4v_mod, gpu, M):
    """Every (sub-group, column) scale a distinct power of two and one +1 code
    per column: with A = 1 each output is exactly the scale of the sub-group
    holding that code (pins s[k/32][n] in both kernels; a power of two times
    1 is exact in fp16)."""
    N, K = 256, 512
    ng = K // G
    s = np.empty((ng, N), np.float16)
    for g in range(ng):
        for n in range(N):
            s[g, n] = 2.0 ** -((g * 7 + n) % 14)
    q = np.full((N, K), 8, np.uint8)
    ks = np.random.default_rng(5).integers(0, K, size=N)
    q[np.arange(N), ks] = 9
    A = np.ones((M, K), np.float16)
    C = _gemm(w4v_mod, gpu, A, q, s)
    want = s[ks // G, np.arange(N)].astype(np.float64)
    assert np.array_equal(C, np.broadcast_to(want, (M, N)))


@pytest.mark.parametrize("N,K", [(2560, 2560), (19456, 2560), (2560, 9728)])
def test_static_weights(w4v_mod, gpu, N, K):
    A, q, s, _ = _case(9, 16, N, K, False, "g32s")
    assert np.array_equal(_gemm(w4v_mod, gpu, A, q, s), _gemm(w4v_mod, gpu, A, q, s, static_weights=True))


def test_batch_invariance(w4v_mod, gpu):
    N, K = 2560, 2560
    A, q, s, _ = _case(6, 32, N, K, False, "g32b")
    full = _gemm(w4v_mod, gpu, A, q, s)
    for m in (1, 7, 16, 21):
        assert np.array_equal(_gemm(w4v_mod, gpu, A[:m], q, s), full[:m]), m
