"""Pins for the oracle's W4A16 dequantization and GEMM.

Definition ("Efficient LLM Challenge Results", sections 3 and 5: 4-bit
W4A16 GPTQ weights with group size 128 and fp16 activations), with the
readings the pages leave open: zero point 8, scales laid out [K/128][N],
C = A @ W^T with W[n][k] = s[k/128][n] * (q[n][k] - 8).

Each pin is a case whose answer is fixed by construction, so that a dropped
term, a wrong sign or index, a transposed operand or a wrong group index
fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

G = 128


def test_half_conversion_all_bit_patterns(oracle_mod):
    """The oracle's own fp16 decoder agrees with numpy's on all 65536 patterns."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    lib = oracle_mod._load()
    got = np.array([lib.oracle_half_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_zero_point_gives_zero(oracle_mod):
    M, N, K = 5, 24, 256
    A = np.random.default_rng(0).standard_normal((M, K)).astype(np.float16)
    q = np.full((N, K), 8, np.uint8)
    s = np.random.default_rng(1).uniform(0.005, 0.02, (K // G, N)).astype(np.float16)
    assert np.all(oracle_mod.w4a16_gemm(A, q, s) == 0.0)


@pytest.mark.parametrize("code,sign", [(9, 1.0), (7, -1.0)])
def test_permutation_weights_pick_columns(oracle_mod, code, sign):
    """q[n][pi(n)] = 8 +- 1, elsewhere 8, unit scales: C[r][n] = +-A[r][pi(n)].
    A non-symmetric permutation catches a transposed weight operand."""
    M, K = 3, 256
    N = K
    rng = np.random.default_rng(2)
    pi = rng.permutation(K)
    q = np.full((N, K), 8, np.uint8)
    q[np.arange(N), pi] = code
    s = np.ones((K // G, N), np.float16)
    A = rng.standard_normal((M, K)).astype(np.float16)
    C = oracle_mod.w4a16_gemm(A, q, s)
    assert np.array_equal(C, sign * A.astype(np.float64)[:, pi])


@pytest.mark.parametrize("G", [128, 32])
def test_group_index_and_scale_orientation(oracle_mod, G):
    """Scales are s[k/G][n]: give every (group, column) a distinct power of two
    and put a single +1 code in one k of one group per column (G = 128, and
    the group size 32 of the compressed-tensors target)."""
    M, N, K = 2, 16, 512
    ng = K // G
    rng = np.random.default_rng(3)
    A = np.ones((M, K), np.float16)
    s = np.empty((ng, N), np.float16)
    for g in range(ng):
        for n in range(N):
            s[g, n] = 2.0 ** -((g * N + n) % 20)
    q = np.full((N, K), 8, np.uint8)
    ks = rng.integers(0, K, size=N)
    q[np.arange(N), ks] = 9
    C = oracle_mod.w4a16_gemm(A, q, s, group=G)
    for n in range(N):
        want = float(s[ks[n] // G, n])
        assert C[0, n] == want and C[1, n] == want


def test_code_range_and_linearity(oracle_mod):
    """Every code c in 0..15 contributes (c - 8) * s * a."""
    M, N, K = 1, 16, 128
    A = np.zeros((M, K), np.float16)
    A[0, 5] = 0.5
    q = np.full((N, K), 8, np.uint8)
    q[:, 5] = np.arange(16)
    s = np.full((1, N), 0.25, np.float16)
    C = oracle_mod.w4a16_gemm(A, q, s)
    assert np.array_equal(C[0], (np.arange(16) - 8) * 0.25 * 0.5)


@pytest.mark.parametrize("G", [128, 32])
def test_zero_table(oracle_mod, G):
    """With a zero table z[k/G][n], W = s * (q - z); q == z gives 0 and q = z + 1 gives s."""
    M, N, K = 2, 8, 256
    rng = np.random.default_rng(4)
    z = rng.integers(0, 15, size=(K // G, N), dtype=np.uint8)
    q = np.repeat(z, G, axis=0).T.copy()               # q[n][k] = z[k/G][n]
    s = np.full((K // G, N), 0.5, np.float16)
    A = rng.standard_normal((M, K)).astype(np.float16)
    assert np.all(oracle_mod.w4a16_gemm(A, q, s, zeros=z, group=G) == 0.0)
    A1 = np.ones((M, K), np.float16)
    C = oracle_mod.w4a16_gemm(A1, q + 1, s, zeros=z, group=G)
    assert np.all(C == 0.5 * K)


def test_exact_rational_small(oracle_mod):
    """Random small case against exact rational arithmetic of the definition."""
    M, N, K = 3, 5, 256
    rng = np.random.default_rng(5)
    A = rng.standard_normal((M, K)).astype(np.float16)
    q = rng.integers(0, 16, (N, K), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float16)
    C = oracle_mod.w4a16_gemm(A, q, s)
    Af = [[Fraction(float(x)) for x in row] for row in A]
    for r in range(M):
        for n in range(N):
            exact = sum(Af[r][k] * Fraction(float(s[k // G, n])) * (int(q[n, k]) - 8) for k in range(K))
            assert abs(C[r, n] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


def test_sampled_matches_full(oracle_mod):
    M, N, K = 4, 40, 384
    rng = np.random.default_rng(6)
    A = rng.standard_normal((M, K)).astype(np.float16)
    q = rng.integers(0, 16, (N, K), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float16)
    C = oracle_mod.w4a16_gemm(A, q, s)
    rows = rng.integers(0, M, 50)
    cols = rng.integers(0, N, 50)
    got = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols)
    assert np.array_equal(got, C[rows, cols])


def test_dequant_matches_gemm_with_identity_activations(oracle_mod):
    """A = I (K x K) returns W^T: the GEMM multiplies by the dequantized matrix."""
    N, K = 16, 128
    rng = np.random.default_rng(7)
    q = rng.integers(0, 16, (N, K), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, (1, N)).astype(np.float16)
    W = oracle_mod.dequant_w4(q, s)
    C = oracle_mod.w4a16_gemm(np.eye(K, dtype=np.float16), q, s)
    assert np.array_equal(C, W.T)
    for n in range(N):
        for k in (0, 17, 127):
            assert W[n, k] == float(s[0, n]) * (int(q[n, k]) - 8)
