"""w4a16_gemm on the GPU against the oracle: max relative error <= 2e-3
(|C - R| / max(|R|, rms R)) against the double-precision definition, on the
small configuration in full and on the 4B-shaped projections on sampled
outputs; plus batch invariance and workspace hygiene."""
import numpy as np
import pytest
import torch

from helpers import GEMM_TOL, gemm_rel_err, to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _gpu_gemm(w4v_mod, gpu, A, q, s, zeros=None, ws=None, static_weights=False):
    N = q.shape[0]
    packed = to_dev(w4v_mod.pack_int4(q), gpu)
    C = w4v_mod.w4a16_gemm(to_dev(A, gpu), packed, to_dev(s, gpu), N,
                           zeros=None if zeros is None else to_dev(zeros, gpu), ws=ws,
                           static_weights=static_weights)
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64)


def test_cfg0_linear(w4v_mod, gpu, oracle_mod):
    """Tiny verify step: M = 16 rows through one 256 -> 512 W4A16 linear."""
    A = inputs.activations(0, 16, 256, "cfg0-a")
    q = inputs.w4_codes(0, 512, 256, "cfg0")
    s = inputs.w4_scales(0, 512, 256, "cfg0")
    C = _gpu_gemm(w4v_mod, gpu, A, q, s)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s)) <= GEMM_TOL


@pytest.mark.parametrize("M,N,K", [(1, 512, 256), (2, 128, 128), (5, 200, 384), (8, 1024, 1024),
                                   (16, 2560, 2560), (17, 520, 640), (21, 768, 1280), (32, 384, 2560),
                                   (16, 2560, 9728), (9, 384, 768), (12, 136, 1664), (31, 264, 1152)])
def test_shapes(w4v_mod, gpu, oracle_mod, M, N, K):
    A = inputs.activations(M, M, K, "shape")
    q = inputs.w4_codes(M, N, K, "shape")
    s = inputs.w4_scales(M, N, K, "shape")
    C = _gpu_gemm(w4v_mod, gpu, A, q, s)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s)) <= GEMM_TOL


@pytest.mark.parametrize("M,N,K", [(16, 512, 512), (3, 272, 640), (24, 400, 3200), (16, 16, 128), (5, 48, 256),
                                   (1, 112, 384), (21, 48, 384)])
def test_zero_points(w4v_mod, gpu, oracle_mod, M, N, K):
    """Per-(group, row) zero points, including odd group counts (a unit
    with a single group at each tile end), a partial last tile, a zero-table
    box narrower than a tile (N < 128) and shorter than a stage (K of one to
    three groups)."""
    A = inputs.activations(3, M, K)
    q = inputs.w4_codes(3, N, K)
    s = inputs.w4_scales(3, N, K)
    z = inputs.w4_zeros(3, N, K)
    C = _gpu_gemm(w4v_mod, gpu, A, q, s, zeros=z)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s, zeros=z)) <= GEMM_TOL


def test_closed_forms_gpu(w4v_mod, gpu):
    """q == 8 gives exactly 0; a +-1 permutation with unit scales gives +-A[:, pi]."""
    M, K = 16, 256
    N = K
    A = inputs.activations(4, M, K)
    s = np.ones((K // 128, N), np.float16)
    C = _gpu_gemm(w4v_mod, gpu, A, np.full((N, K), 8, np.uint8), s)
    assert np.all(C == 0)
    pi = np.random.default_rng(4).permutation(K)
    q = np.full((N, K), 8, np.uint8)
    q[np.arange(N), pi] = 7
    C = _gpu_gemm(w4v_mod, gpu, A, q, s)
    assert np.array_equal(C, -A.astype(np.float64)[:, pi])


@pytest.mark.parametrize("M,N,K,zeros", [(16, 2560, 2560, False), (16, 7680, 2560, False), (16, 2560, 9728, False),
                                         (5, 200, 384, False), (24, 400, 3200, True), (16, 19456, 2560, False)])
def test_static_weights(w4v_mod, gpu, oracle_mod, M, N, K, zeros):
    """With the static-weights promise the first weight stages are loaded and
    dequantized before the previous kernel ends; the arithmetic is the same,
    so the result equals the plain call bit for bit (both work splits)."""
    A = inputs.activations(9, M, K, "static")
    q = inputs.w4_codes(9, N, K, "static")
    s = inputs.w4_scales(9, N, K, "static")
    z = inputs.w4_zeros(9, N, K, "static") if zeros else None
    plain = _gpu_gemm(w4v_mod, gpu, A, q, s, zeros=z)
    early = _gpu_gemm(w4v_mod, gpu, A, q, s, zeros=z, static_weights=True)
    assert np.array_equal(plain, early)
    if N * K <= 2560 * 2560:
        assert gemm_rel_err(early, oracle_mod.w4a16_gemm(A, q, s, zeros=z)) <= GEMM_TOL


def test_batch_invariance(w4v_mod, gpu):
    """For M <= 32 every output element comes from the same arithmetic, so the
    rows of a small-M call equal the same rows of a larger call bit for bit."""
    N, K = 2560, 2560
    A = inputs.activations(6, 32, K)
    q = inputs.w4_codes(6, N, K)
    s = inputs.w4_scales(6, N, K)
    full = _gpu_gemm(w4v_mod, gpu, A, q, s)
    for m in (1, 7, 16, 21):
        part = _gpu_gemm(w4v_mod, gpu, A[:m], q, s)
        assert np.array_equal(part, full[:m]), m


def test_workspace_reuse_is_clean(w4v_mod, gpu):
    M, N, K = 16, 2560, 9728
    A = inputs.activations(7, M, K)
    q = inputs.w4_codes(7, N, K)
    s = inputs.w4_scales(7, N, K)
    ws = w4v_mod.workspace(w4v_mod.w4a16_workspace_bytes(M, N, K), gpu)
    a = _gpu_gemm(w4v_mod, gpu, A, q, s, ws=ws)
    b = _gpu_gemm(w4v_mod, gpu, A, q, s, ws=ws)
    assert np.array_equal(a, b)
    n_tiles = -(-N // 128)
    counters = ws.cpu().numpy()[-(((n_tiles * 4 + 255) // 256) * 256):]
    assert np.all(counters == 0)
    assert w4v_mod.get_status() == 0


@pytest.mark.parametrize("zeros", [False, True], ids=["sym", "zeros"])
@pytest.mark.parametrize("M", [16, 21, 32])
@pytest.mark.parametrize("proj", inputs.LAYER_PROJS, ids=lambda p: p.name)
def test_layer_projection_sampled(w4v_mod, gpu, oracle_mod, proj, M, zeros):
    """The 4B-shaped projections at the verify sizes of K = 15 drafts (M = 16),
    of the runner-up's constant K = 20 (M = 21) and at 32 rows, each with and
    without a zero table (gate_up takes the stream-K split, the others the
    cluster split): 4000 sampled outputs plus two full output rows against
    the oracle."""
    A = inputs.activations(1, M, proj.K, 0, proj.name)
    q, s = inputs.layer_weights(1, 0, proj)
    z = inputs.w4_zeros(1, proj.N, proj.K, proj.name) if zeros else None
    C = _gpu_gemm(w4v_mod, gpu, A, q, s, zeros=z)
    r = np.random.default_rng(M)
    rows = r.integers(0, M, 4000).astype(np.int32)
    cols = r.integers(0, proj.N, 4000).astype(np.int32)
    rows = np.concatenate([rows, np.zeros(proj.N, np.int32), np.full(proj.N, M - 1, np.int32)])
    cols = np.concatenate([cols, np.arange(proj.N, dtype=np.int32), np.arange(proj.N, dtype=np.int32)])
    R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols, zeros=z)
    assert gemm_rel_err(C[rows, cols], R) <= GEMM_TOL


# ---------------------------------------------------------------- prefill (M > 32)
@pytest.mark.parametrize("M,N,K", [(33, 512, 256), (64, 128, 128), (128, 2560, 2560), (200, 520, 640),
                                   (256, 1024, 1280), (300, 384, 9728), (768, 2560, 512)])
def test_prefill_shapes(w4v_mod, gpu, oracle_mod, M, N, K):
    A = inputs.activations(M, M, K, "prefill")
    q = inputs.w4_codes(M, N, K, "prefill")
    s = inputs.w4_scales(M, N, K, "prefill")
    C = _gpu_gemm(w4v_mod, gpu, A, q, s)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s)) <= GEMM_TOL


@pytest.mark.parametrize("M,N,K", [(96, 256, 512), (2048, 2560, 512)])
def test_prefill_zero_points(w4v_mod, gpu, oracle_mod, M, N, K):
    """Zero tables on the prefill kernel: a few row slices, and 152 whole
    tiles (each accumulator half from its own issuer) plus 32 slices."""
    A = inputs.activations(8, M, K)
    q = inputs.w4_codes(8, N, K)
    s = inputs.w4_scales(8, N, K)
    z = inputs.w4_zeros(8, N, K)
    C = _gpu_gemm(w4v_mod, gpu, A, q, s, zeros=z)
    assert gemm_rel_err(C, oracle_mod.w4a16_gemm(A, q, s, zeros=z)) <= GEMM_TOL


@pytest.mark.parametrize("M", [2048, 8192])
@pytest.mark.parametrize("proj", inputs.LAYER_PROJS, ids=lambda p: p.name)
def test_prefill_layer_projection_sampled(w4v_mod, gpu, oracle_mod, proj, M):
    """The 4B-shaped projections at prefill sizes (2048 and 8192 rows): 3000
    sampled outputs plus one full output row and one full column."""
    A = inputs.activations(2, M, proj.K, 0, proj.name, "prefill")
    q, s = inputs.layer_weights(2, 0, proj)
    C = _gpu_gemm(w4v_mod, gpu, A, q, s)
    r = np.random.default_rng(M)
    rows = r.integers(0, M, 3000).astype(np.int32)
    cols = r.integers(0, proj.N, 3000).astype(np.int32)
    rows = np.concatenate([rows, np.full(proj.N, M - 1, np.int32), np.arange(0, M, max(1, M // 256), dtype=np.int32)])
    cols = np.concatenate([cols, np.arange(proj.N, dtype=np.int32),
                           np.full(len(range(0, M, max(1, M // 256))), proj.N - 1, np.int32)])
    R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols)
    assert gemm_rel_err(C[rows, cols], R) <= GEMM_TOL


@pytest.mark.parametrize("M,N,K", [(300, 2560, 2560), (2048, 2560, 9728), (2048, 2560, 2560),
                                   (700, 2560, 1024)])
def test_prefill_split_tiles_deterministic_and_clean(w4v_mod, gpu, oracle_mod, M, N, K):
    """Shapes whose last wave is mostly empty: the first splits the k range
    of tiles between CTAs (fp32 partials added by the last contributor in
    CTA order), o and down at 2048 rows cut the last wave's 8 tiles into 32
    slices of 64 rows, and 60 tiles with a ragged last row of tiles (700
    rows) become 120 slices of 128: repeated calls on one workspace are
    bit-identical, the arrival counters are left at zero, and sampled
    outputs match the oracle."""
    A = inputs.activations(M, M, K, "split")
    q = inputs.w4_codes(M, N, K, "split")
    s = inputs.w4_scales(M, N, K, "split")
    ws = w4v_mod.workspace(w4v_mod.w4a16_workspace_bytes(M, N, K), gpu)
    a = _gpu_gemm(w4v_mod, gpu, A, q, s, ws=ws)
    b = _gpu_gemm(w4v_mod, gpu, A, q, s, ws=ws)
    assert np.array_equal(a, b)
    tiles = -(-N // 128) * -(-M // 256)
    counters = ws.cpu().numpy()[-(((tiles * 4 + 255) // 256) * 256):]
    assert np.all(counters == 0)
    r = np.random.default_rng(M + N)
    rows = r.integers(0, M, 3000).astype(np.int32)
    cols = r.integers(0, N, 3000).astype(np.int32)
    R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols)
    assert gemm_rel_err(a[rows, cols], R) <= GEMM_TOL
    assert w4v_mod.get_status() == 0


@pytest.mark.parametrize("M", [16, 21, 32])
def test_back_to_back_layer_launches_clean_and_deterministic(w4v_mod, gpu, M):
    """The 4B layer's projections launched back to back many times with
    static weights (each launch's set-up overlapping the previous one, as in
    the verify step): no kernel may give up a bounded wait (device status
    stays clear) and every launch must reproduce the first one's outputs bit
    for bit.  A barrier whose phases a waiter can skip shows up here as a
    timeout or as a changed output; M = 21 and 32 run two accumulator sets
    per tile, M = 16 four."""
    g = torch.Generator(device=gpu)
    g.manual_seed(71 + M)
    projs = []
    for p in inputs.LAYER_PROJS:
        packed = torch.randint(0, 256, (w4v_mod.packed_bytes(p.N, p.K),), generator=g, device=gpu,
                               dtype=torch.uint8)
        sc = (torch.rand((p.K // 128, p.N), generator=g, device=gpu) * 0.015 + 0.005).half()
        A = torch.randn((M, p.K), generator=g, device=gpu).half()
        ws = w4v_mod.workspace(w4v_mod.w4a16_workspace_bytes(M, p.N, p.K), gpu)
        projs.append((p, packed, sc, A, ws))
    assert w4v_mod.get_status() == 0
    ref = [w4v_mod.w4a16_gemm(A, packed, sc, p.N, ws=ws, static_weights=True).clone()
           for (p, packed, sc, A, ws) in projs]
    outs = [torch.empty_like(r) for r in ref]
    for _ in range(100):
        for (p, packed, sc, A, ws), C in zip(projs, outs):
            w4v_mod.w4a16_gemm(A, packed, sc, p.N, out=C, ws=ws, static_weights=True)
    torch.cuda.synchronize()
    assert w4v_mod.get_status() == 0
    for r, C in zip(ref, outs):
        assert torch.equal(r, C)


@pytest.mark.parametrize("zeros", [False, True], ids=["sym", "zeros"])
def test_batch_invariant_blocks(w4v_mod, gpu, oracle_mod, zeros):
    """W4V_BATCH_INVARIANT: 8 sequences x 16 verify positions (128 rows) in
    one call give each sequence's rows bit for bit what that sequence's own
    16-row call gives (and each row what a 1-row call gives), so a batched
    verify never changes an accepted token; sampled outputs meet the oracle
    bound.  Without the flag 128 rows take the prefill kernel, whose
    rounding differs."""
    N, K = 2560, 2560
    A = inputs.activations(81, 128, K, "binv")
    q = inputs.w4_codes(81, N, K, "binv")
    s = inputs.w4_scales(81, N, K, "binv")
    z = inputs.w4_zeros(81, N, K, "binv") if zeros else None
    packed = to_dev(w4v_mod.pack_int4(q), gpu)
    sd = to_dev(s, gpu)
    zd = None if z is None else to_dev(z, gpu)
    Ad = to_dev(A, gpu)
    C128 = w4v_mod.w4a16_gemm(Ad, packed, sd, N, zeros=zd, batch_invariant=True).cpu().numpy()
    for b in range(8):
        C16 = w4v_mod.w4a16_gemm(Ad[16 * b:16 * b + 16].contiguous(), packed, sd, N, zeros=zd).cpu().numpy()
        assert np.array_equal(C16, C128[16 * b:16 * b + 16]), b
    for m in (0, 45, 127):
        C1 = w4v_mod.w4a16_gemm(Ad[m:m + 1].contiguous(), packed, sd, N, zeros=zd).cpu().numpy()
        assert np.array_equal(C1[0], C128[m]), m
    r = np.random.default_rng(81)
    rows = r.integers(0, 128, 3000).astype(np.int32)
    cols = r.integers(0, N, 3000).astype(np.int32)
    R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols, zeros=z)
    assert gemm_rel_err(C128.astype(np.float64)[rows, cols], R) <= GEMM_TOL
    assert w4v_mod.get_status() == 0
