"""w4a16_gemm_grouped on the GPU against the oracle.

A grouped launch streams several independent W4A16 products through one
pipeline ("Efficient LLM Challenge Results", section 2 "Where the time goes":
decode is bound by reading the weights, so the start-up of one launch per
few-MB projection is pure loss).  Every output of every problem must meet the
same bound as w4a16_gemm: max |C - R| / max(|R|, rms R) <= 2e-3 against the
double-precision oracle.  The work split crosses tile and problem
boundaries, so the cases mix ragged shapes (partial tiles, odd group counts,
N below one tile, K of one or two groups), many problems, zero points, group
size 32 and M from 1 to 32."""
import numpy as np
import pytest
import torch

from helpers import GEMM_TOL, gemm_rel_err, to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _host(seed, M, shapes, zeros=False, group=128, tag="grouped"):
    out = []
    for i, (N, K) in enumerate(shapes):
        A = inputs.activations(seed, M, K, tag, i)
        q = inputs.w4_codes(seed, N, K, tag, i)
        s = inputs.w4_scales(seed, N, K, tag, i, group=group)
        z = inputs.w4_zeros(seed, N, K, tag, i, group=group) if zeros else None
        out.append((A, q, s, z))
    return out


def _device(w4v_mod, gpu, host):
    dev = []
    for (A, q, s, z) in host:
        dev.append((to_dev(A, gpu), to_dev(w4v_mod.pack_int4(q), gpu), to_dev(s, gpu),
                    None if z is None else to_dev(z, gpu),
                    torch.empty((A.shape[0], q.shape[0]), dtype=torch.float16, device=gpu)))
    return dev


def _run(grouped, static_weights=False):
    outs = grouped(static_weights=static_weights)
    torch.cuda.synchronize()
    return [C.cpu().numpy().astype(np.float64) for C in outs]


def _check_oracle(oracle_mod, host, outs, group=128):
    for i, ((A, q, s, z), C) in enumerate(zip(host, outs)):
        R = oracle_mod.w4a16_gemm(A, q, s, zeros=z, group=group)
        assert gemm_rel_err(C, R) <= GEMM_TOL, i


MIXED = [(512, 256), (200, 384), (2560, 1280), (48, 128), (1024, 1024), (136, 1664), (16, 256), (2048, 640)]


@pytest.mark.parametrize("M", [1, 5, 16, 21, 32])
def test_mixed_shapes(w4v_mod, gpu, oracle_mod, M):
    """Eight problems of mixed sizes (187 work units over the SMs, so CTAs
    start and end inside tiles and across problems) against the oracle."""
    host = _host(M, M, MIXED)
    g = w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host))
    _check_oracle(oracle_mod, host, _run(g))
    assert w4v_mod.get_status() == 0


def test_fewer_units_than_sms(w4v_mod, gpu, oracle_mod):
    """Three small problems (9 units): one unit per CTA, every tile split."""
    host = _host(3, 16, [(256, 384), (128, 512), (64, 256)])
    g = w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host))
    _check_oracle(oracle_mod, host, _run(g))


def test_many_problems(w4v_mod, gpu, oracle_mod):
    """300 small problems of random shapes: table lookups across hundreds of
    problem boundaries inside single CTAs."""
    r = np.random.default_rng(300)
    shapes = [(int(8 * r.integers(1, 64)), int(128 * r.integers(1, 9))) for _ in range(300)]
    host = _host(300, 16, shapes, tag="many")
    g = w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host))
    _check_oracle(oracle_mod, host, _run(g))
    assert w4v_mod.get_status() == 0


@pytest.mark.parametrize("M", [3, 16, 21])
def test_zero_points(w4v_mod, gpu, oracle_mod, M):
    """Zero tables (group 128), including a box narrower than a tile (N < 128)
    and shorter than a stage (K of one to three groups)."""
    shapes = [(16, 128), (48, 256), (112, 384), (512, 512), (272, 640), (400, 3200), (2560, 1280)]
    host = _host(11 + M, M, shapes, zeros=True, tag="zeros")
    g = w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host))
    _check_oracle(oracle_mod, host, _run(g))


@pytest.mark.parametrize("zeros", [False, True])
@pytest.mark.parametrize("M", [1, 16, 21])
def test_group32(w4v_mod, gpu, oracle_mod, M, zeros):
    shapes = [(512, 256), (200, 384), (2560, 1280), (48, 128), (136, 1664)] if not zeros else \
             [(16, 128), (48, 256), (512, 512), (272, 640), (2560, 1280)]
    host = _host(21 + M, M, shapes, zeros=zeros, group=32, tag="g32")
    g = w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host), group=32)
    _check_oracle(oracle_mod, host, _run(g), group=32)


def test_batch_invariance(w4v_mod, gpu):
    """The work split depends on the shapes only, so the rows of a small-M
    grouped launch equal the same rows of a 32-row launch bit for bit."""
    host32 = _host(41, 32, MIXED)
    full = _run(w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host32)))
    for m in (1, 7, 16, 21):
        host = [(A[:m], q, s, z) for (A, q, s, z) in host32]
        part = _run(w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host)))
        for i in range(len(host)):
            assert np.array_equal(part[i], full[i][:m]), (m, i)


@pytest.mark.parametrize("M", [16, 21])
def test_repeated_launches_clean_and_deterministic(w4v_mod, gpu, M):
    """50 launches back to back with static weights on one workspace: bit
    for bit the first launch's outputs, counters back at zero, no kernel gave
    up a bounded wait."""
    host = _host(51, M, MIXED)
    dev = _device(w4v_mod, gpu, host)
    g = w4v_mod.GroupedGemm(dev)
    first = _run(g, static_weights=True)
    for _ in range(50):
        g(static_weights=True)
    torch.cuda.synchronize()
    assert w4v_mod.get_status() == 0
    again = [C.cpu().numpy().astype(np.float64) for (_, _, _, _, C) in dev]
    for a, b in zip(first, again):
        assert np.array_equal(a, b)
    # the arrival counters (after the partial tiles) are back at zero
    tiles = g.handle.tiles
    counters = g.ws.cpu().numpy()[-(((tiles * 4 + 255) // 256) * 256):]
    assert np.all(counters == 0)


@pytest.mark.parametrize("zeros", [False, True])
@pytest.mark.parametrize("M", [16, 21, 32])
def test_layer_set_sampled(w4v_mod, gpu, oracle_mod, M, zeros):
    """The 4B-shaped layer set (qkv, o, gate_up, down) in one launch at the
    verify sizes of K = 15 and K = 20 drafts (and 32 rows): 3000 sampled
    outputs and the first and last full output rows of every projection
    against the oracle, with and without zero tables."""
    host = []
    for i, p in enumerate(inputs.LAYER_PROJS):
        A = inputs.activations(61, M, p.K, p.name, "grouped-layer")
        q, s = inputs.layer_weights(61, 0, p)
        z = inputs.w4_zeros(61, p.N, p.K, p.name) if zeros else None
        host.append((A, q, s, z))
    g = w4v_mod.GroupedGemm(_device(w4v_mod, gpu, host))
    outs = _run(g, static_weights=True)
    r = np.random.default_rng(M)
    for (A, q, s, z), C in zip(host, outs):
        N = q.shape[0]
        rows = r.integers(0, M, 3000).astype(np.int32)
        cols = r.integers(0, N, 3000).astype(np.int32)
        rows = np.concatenate([rows, np.zeros(N, np.int32), np.full(N, M - 1, np.int32)])
        cols = np.concatenate([cols, np.arange(N, dtype=np.int32), np.arange(N, dtype=np.int32)])
        R = oracle_mod.w4a16_gemm_sampled(A, q, s, rows, cols, zeros=z)
        assert gemm_rel_err(C[rows, cols], R) <= GEMM_TOL
    assert w4v_mod.get_status() == 0
