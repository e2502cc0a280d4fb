"""The oracle's gated delta recurrence against closed forms.

The recurrence (Yang et al., "Gated Delta Networks", reference [12] of
"Efficient LLM Challenge Results"; the state a rejected draft must not
touch, section 3 and "DFlash K=15 for Qwen3.5-4B on a single A10G", "What
transfers"):  S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
o_t = S_t q_t.  Basis keys and power-of-two gates make every case exact, so
a wrong index orientation, a dropped erase term, a wrong sign, a wrong
ordering of update and read-out, or a stale final state fails one of them.
"""
import numpy as np
import pytest


def _e(d, j):
    x = np.zeros(d)
    x[j] = 1.0
    return x


def test_no_write_is_pure_decay(oracle_mod):
    """beta = 0: S_T = (prod alpha) S0 and o_t = S_t q_t."""
    rng = np.random.default_rng(1)
    H, T, dk, dv = 2, 4, 8, 6
    S0 = rng.standard_normal((H, dv, dk))
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    alpha = np.array([[0.5, 1.0], [0.25, 0.5], [1.0, 0.125], [0.5, 0.5]])
    beta = np.zeros((T, H))
    o, S = oracle_mod.gdn_recurrence(S0, q, k, v, alpha, beta)
    decay = np.cumprod(alpha, axis=0)
    for h in range(H):
        assert np.array_equal(S[h], decay[-1, h] * S0[h])
        for t in range(T):
            assert np.allclose(o[t, h], decay[t, h] * S0[h] @ q[t, h], rtol=1e-14, atol=0)


def test_delta_rule_writes_value_under_key(oracle_mod):
    """alpha = beta = 1, k = e_j: column j of S becomes v exactly, the other
    columns are untouched (pins S[v index][k index] and the erase term)."""
    rng = np.random.default_rng(2)
    dk, dv = 8, 5
    S0 = rng.integers(-8, 8, size=(1, dv, dk)).astype(np.float64)
    j = 3
    v = rng.integers(-8, 8, size=(1, 1, dv)).astype(np.float64)
    o, S = oracle_mod.gdn_recurrence(S0, _e(dk, 0).reshape(1, 1, dk), _e(dk, j).reshape(1, 1, dk), v,
                                     np.ones((1, 1)), np.ones((1, 1)))
    want = S0[0].copy()
    want[:, j] = v[0, 0]
    assert np.array_equal(S[0], want)
    assert np.array_equal(o[0, 0], want[:, 0])


def test_partial_write_and_decay(oracle_mod):
    """k = e_j, beta = 1/4, alpha = 1/2: column j -> alpha (1 - beta) S0_j + beta v,
    other columns -> alpha S0 (the decay multiplies the erased state, not the write)."""
    dk, dv, j = 4, 3, 1
    S0 = np.arange(dv * dk, dtype=np.float64).reshape(1, dv, dk)
    v = np.array([[[4.0, -8.0, 2.0]]])
    o, S = oracle_mod.gdn_recurrence(S0, _e(dk, j).reshape(1, 1, dk), _e(dk, j).reshape(1, 1, dk), v,
                                     np.full((1, 1), 0.5), np.full((1, 1), 0.25))
    want = 0.5 * S0[0]
    want[:, j] = 0.5 * 0.75 * S0[0, :, j] + 0.25 * v[0, 0]
    assert np.array_equal(S[0], want)
    assert np.array_equal(o[0, 0], want[:, j])          # read-out after the update


def test_output_reads_the_updated_state(oracle_mod):
    """S0 = 0, q = k = e_j: o_0 = v_0 (an output taken before the update would be 0)."""
    dk, dv = 4, 4
    v = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    o, _ = oracle_mod.gdn_recurrence(np.zeros((1, dv, dk)), _e(dk, 2).reshape(1, 1, dk),
                                     _e(dk, 2).reshape(1, 1, dk), v, np.ones((1, 1)), np.ones((1, 1)))
    assert np.array_equal(o[0, 0], v[0, 0])


def test_orthogonal_keys_fill_columns(oracle_mod):
    """Writes under distinct basis keys land in their own columns, in any order."""
    dk, dv, T = 6, 3, 4
    keys = [4, 0, 5, 2]
    v = np.arange(T * dv, dtype=np.float64).reshape(T, 1, dv) + 1
    k = np.stack([_e(dk, j) for j in keys]).reshape(T, 1, dk)
    one = np.ones((T, 1))
    _, S = oracle_mod.gdn_recurrence(np.zeros((1, dv, dk)), k, k, v, one, one)
    perm = [2, 0, 3, 1]
    _, S2 = oracle_mod.gdn_recurrence(np.zeros((1, dv, dk)), k[perm], k[perm], v[perm], one, one)
    for t, j in enumerate(keys):
        assert np.array_equal(S[0][:, j], v[t, 0])
    assert np.array_equal(S, S2)


@pytest.mark.parametrize("n", [0, 1, 5, 15])
def test_prefix_replay_equals_the_run(oracle_mod, n):
    """Rolling back = replaying the accepted prefix: running positions 0..n from
    S0 gives the same outputs and the same state as the first n+1 steps of the
    full run, and running the rest from that state continues the full run."""
    rng = np.random.default_rng(n)
    H, T, dk, dv = 2, 16, 16, 8
    S0 = rng.standard_normal((H, dv, dk))
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    alpha = rng.uniform(0.5, 1.0, (T, H))
    beta = rng.uniform(0.0, 1.0, (T, H))
    o, S = oracle_mod.gdn_recurrence(S0, q, k, v, alpha, beta)
    o1, S1 = oracle_mod.gdn_recurrence(S0, q[:n + 1], k[:n + 1], v[:n + 1], alpha[:n + 1], beta[:n + 1])
    assert np.array_equal(o1, o[:n + 1])
    if n + 1 < T:
        o2, S2 = oracle_mod.gdn_recurrence(S1, q[n + 1:], k[n + 1:], v[n + 1:], alpha[n + 1:], beta[n + 1:])
        assert np.array_equal(o2, o[n + 1:])
        assert np.array_equal(S2, S)
    else:
        assert np.array_equal(S1, S)
