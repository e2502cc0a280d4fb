"""spec_accept on the GPU against the oracle: bit-exact accepted lengths and
emitted tokens ("Efficient LLM Challenge Results", section 3)."""
import numpy as np
import pytest

from conftest import read_golden
from helpers import to_dev

pytestmark = pytest.mark.gpu


def _ints(field):
    return [int(x) for x in field.split()] if field.strip() else []


def test_golden_cases_gpu(w4v_mod, gpu, oracle_mod):
    for d, t, n, emitted in read_golden("accept_cases.txt"):
        d, t, n = _ints(d), _ints(t), int(n)
        T = to_dev(np.array([t], np.int32), gpu)
        D = to_dev(np.array([d], np.int32).reshape(1, len(d)), gpu)
        ng, tok = w4v_mod.spec_accept(T, D)
        assert int(ng.cpu()[0]) == n, (d, t)
        assert list(tok.cpu().numpy()[0, : n + 1]) == _ints(emitted)
        assert all(x == -1 for x in tok.cpu().numpy()[0, n + 1:])


@pytest.mark.parametrize("K", [0, 1, 15, 20, 31, 32, 33, 100, 1024])
def test_random_batches_match_oracle(w4v_mod, gpu, oracle_mod, K):
    from speculative_decoding_verify_w4a16_gb300 import inputs
    B, V = 777, 50
    r = np.random.default_rng(K)
    t = r.integers(0, V, size=(B, K + 1)).astype(np.int32)
    d, _ = inputs.drafts_padded(K + 3, t, V, 0.8)
    flip = r.random(size=d.shape) < 0.02
    d = np.where(flip, -1, d).astype(np.int32)
    n_o, tok_o = oracle_mod.spec_accept(t, d)
    n_g, tok_g = w4v_mod.spec_accept(to_dev(t, gpu), to_dev(d, gpu))
    assert np.array_equal(n_g.cpu().numpy(), n_o)
    assert np.array_equal(tok_g.cpu().numpy(), tok_o)
    assert w4v_mod.get_status() == 0
