"""gdn_verify / gdn_commit on the GPU against the oracle's gated delta
recurrence (the Gated DeltaNet state a rejected draft must not touch:
"Efficient LLM Challenge Results", section 3, runner-up paragraph; "DFlash
K=15 for Qwen3.5-4B on a single A10G", "What transfers").

Tolerances follow from the arithmetic: the kernels run the recurrence in
fp32, the oracle in double.  With |k| = 1, 0 < alpha <= 1, 0 <= beta <= 1
the map S -> alpha S (I - beta k k^T) does not grow S, so each step adds at
most about (dk + 3) fp32 roundings relative to the state's size: over T <= 21
steps that is below T (dk + 3) 2^-24 ~ 1.6e-4, the state's bound.  The
outputs are rounded to fp16 (2^-11 relative) on top: 1e-3.
"""
import numpy as np
import pytest
import torch

from helpers import to_dev
from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu
STATE_TOL = 1.6e-4
OUT_TOL = 1e-3


def _rel(C, R):
    R = np.asarray(R, np.float64)
    scale = max(float(np.max(np.abs(R))), 1e-30)
    return float(np.max(np.abs(np.asarray(C, np.float64) - R))) / scale


def _block(seed, B, T, H, dv, dk=128):
    r = inputs.rng(seed, "gdn", B, T, H, dv)
    S0 = r.standard_normal((B, H, dv, dk)).astype(np.float32)
    q = r.standard_normal((B, T, H, dk))
    k = r.standard_normal((B, T, H, dk))
    q = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float16)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float16)
    v = r.standard_normal((B, T, H, dv)).astype(np.float16)
    alpha = r.uniform(0.5, 1.0, (B, T, H)).astype(np.float32)
    beta = r.uniform(0.0, 1.0, (B, T, H)).astype(np.float32)
    return S0, q, k, v, alpha, beta


def _oracle(oracle_mod, S0, q, k, v, alpha, beta, b, T=None):
    T = q.shape[1] if T is None else T
    return oracle_mod.gdn_recurrence(S0[b], q[b, :T], k[b, :T], v[b, :T], alpha[b, :T], beta[b, :T])


@pytest.mark.parametrize("B,T,H,dv", [(1, 16, 4, 128), (3, 21, 2, 64), (2, 1, 3, 32), (1, 32, 1, 256),
                                      (2, 16, 32, 128)])
def test_verify_outputs(w4v_mod, gpu, oracle_mod, B, T, H, dv):
    S0, q, k, v, alpha, beta = _block(B * 100 + T, B, T, H, dv)
    Sd = to_dev(S0, gpu)
    o = w4v_mod.gdn_verify(Sd, to_dev(q, gpu), to_dev(k, gpu), to_dev(v, gpu), to_dev(alpha, gpu), to_dev(beta, gpu))
    torch.cuda.synchronize()
    o = o.cpu().numpy()
    assert np.array_equal(Sd.cpu().numpy(), S0)          # verify never writes the state
    for b in range(B):
        o_ref, _ = _oracle(oracle_mod, S0, q, k, v, alpha, beta, b)
        assert _rel(o[b], o_ref) <= OUT_TOL, b


@pytest.mark.parametrize("B,T,H,dv", [(4, 16, 2, 128), (3, 21, 3, 64), (2, 1, 1, 32)])
def test_commit_rolls_back_rejected_positions(w4v_mod, gpu, oracle_mod, B, T, H, dv):
    """The committed state equals the oracle's state after positions 0..n[b]
    only; n spans none accepted, some, all, and out-of-range values (clamped)."""
    S0, q, k, v, alpha, beta = _block(7 + T, B, T, H, dv)
    n = np.array([0, T // 2, T - 1, T + 5][:B], np.int32)
    Sd = to_dev(S0, gpu)
    w4v_mod.gdn_commit(Sd, to_dev(k, gpu), to_dev(v, gpu), to_dev(alpha, gpu), to_dev(beta, gpu), to_dev(n, gpu))
    torch.cuda.synchronize()
    S = Sd.cpu().numpy()
    for b in range(B):
        steps = min(int(n[b]), T - 1) + 1
        _, S_ref = _oracle(oracle_mod, S0, q, k, v, alpha, beta, b, steps)
        assert _rel(S[b], S_ref) <= STATE_TOL, b


def test_verify_then_commit_equals_plain_decoding(w4v_mod, gpu, oracle_mod):
    """A speculative block verified then committed with n accepted equals
    n + 1 single-position steps (verify of T = 1 then commit of n = 0, the
    plain decoding path): outputs of the accepted positions and final state."""
    B, T, H, dv = 2, 16, 2, 64
    S0, q, k, v, alpha, beta = _block(11, B, T, H, dv)
    n = np.array([6, 15], np.int32)
    d = lambda a: to_dev(a, gpu)
    Sd = d(S0)
    o_blk = w4v_mod.gdn_verify(Sd, d(q), d(k), d(v), d(alpha), d(beta))
    w4v_mod.gdn_commit(Sd, d(k), d(v), d(alpha), d(beta), d(n))
    Ss = d(S0)
    o_seq = []
    zero = d(np.zeros(B, np.int32))
    for t in range(T):
        sl = lambda a: d(np.ascontiguousarray(a[:, t:t + 1]))
        o_seq.append(w4v_mod.gdn_verify(Ss, sl(q), sl(k), sl(v), sl(alpha), sl(beta)))
        if t <= n.min():
            w4v_mod.gdn_commit(Ss, sl(k), sl(v), sl(alpha), sl(beta), zero)
    torch.cuda.synchronize()
    o_blk = o_blk.cpu().numpy()
    o_seq = np.concatenate([x.cpu().numpy() for x in o_seq], axis=1)
    m = int(n.min())
    # the first m+1 positions see the same states either way
    assert _rel(o_blk[:, : m + 1], o_seq[:, : m + 1]) <= OUT_TOL
    # sequence 0 (n = 6) committed exactly positions 0..6 both ways
    assert _rel(Sd.cpu().numpy()[0], Ss.cpu().numpy()[0]) <= STATE_TOL


def test_delta_rule_closed_form_gpu(w4v_mod, gpu):
    """alpha = beta = 1 and a basis key e_j: the committed state's column j is
    exactly v and every other column is unchanged; the output under query
    e_j is v (exact in fp32: every product involves a 0 or a 1)."""
    B, T, H, dv, dk = 1, 1, 1, 32, 128
    S0 = np.arange(B * H * dv * dk, dtype=np.float32).reshape(B, H, dv, dk) / 64
    j = 77
    k = np.zeros((B, T, H, dk), np.float16)
    k[..., j] = 1
    v = (np.arange(dv, dtype=np.float32) - 9).astype(np.float16).reshape(B, T, H, dv)
    one = np.ones((B, T, H), np.float32)
    d = lambda a: to_dev(a, gpu)
    Sd = d(S0)
    o = w4v_mod.gdn_verify(Sd, d(k), d(k), d(v), d(one), d(one))
    w4v_mod.gdn_commit(Sd, d(k), d(v), d(one), d(one), d(np.zeros(B, np.int32)))
    torch.cuda.synchronize()
    want = S0.copy()
    want[0, 0, :, j] = v[0, 0, 0].astype(np.float32)
    assert np.array_equal(Sd.cpu().numpy(), want)
    assert np.array_equal(o.cpu().numpy()[0, 0, 0], v[0, 0, 0])


@pytest.mark.parametrize("B,T,T_prev,H,dv", [(2, 16, 16, 2, 128), (3, 21, 5, 3, 64), (1, 1, 1, 1, 32),
                                             (2, 16, 0, 2, 64), (4, 8, 21, 2, 32)])
def test_step_equals_commit_then_verify(w4v_mod, gpu, oracle_mod, B, T, T_prev, H, dv):
    """gdn_step (commit of the previous block, verify of the next, one launch)
    gives bit for bit the state and outputs of gdn_commit followed by
    gdn_verify, and the oracle's within the recurrence's bounds; n spans none
    accepted, some, all and out of range."""
    d = lambda a: to_dev(a, gpu)
    S0, q, k, v, alpha, beta = _block(300 + T, B, T, H, dv)
    if T_prev > 0:
        _, _, kp, vp, ap, bp = _block(400 + T_prev, B, T_prev, H, dv)
        n = np.array([0, T_prev // 2, T_prev - 1, T_prev + 3][:B], np.int32)
    Sa, Sb = d(S0), d(S0)
    if T_prev > 0:
        w4v_mod.gdn_commit(Sa, d(kp), d(vp), d(ap), d(bp), d(n))
    o_ref = w4v_mod.gdn_verify(Sa, d(q), d(k), d(v), d(alpha), d(beta))
    prev = (d(kp), d(vp), d(ap), d(bp), d(n)) if T_prev > 0 else None
    o = w4v_mod.gdn_step(Sb, prev, d(q), d(k), d(v), d(alpha), d(beta))
    torch.cuda.synchronize()
    assert torch.equal(Sa, Sb)
    assert torch.equal(o_ref, o)
    if T_prev == 0:
        assert np.array_equal(Sb.cpu().numpy(), S0)      # nothing to commit: state untouched
    for b in range(B):
        S_b = S0[b]
        if T_prev > 0:
            steps = min(int(n[b]), T_prev - 1) + 1
            _, S_b = oracle_mod.gdn_recurrence(S0[b], np.zeros_like(kp[b, :steps]), kp[b, :steps], vp[b, :steps],
                                               ap[b, :steps], bp[b, :steps])
            assert _rel(Sb.cpu().numpy()[b], S_b) <= STATE_TOL, b
        o_or, _ = oracle_mod.gdn_recurrence(S_b, q[b], k[b], v[b], alpha[b], beta[b])
        assert _rel(o.cpu().numpy()[b], o_or) <= OUT_TOL + STATE_TOL, b
