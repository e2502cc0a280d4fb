"""The lm_head entry point for callers that cannot allocate device memory.

Some callers cannot provide a workspace -- a plugin inside another inference
engine that may not allocate while it executes, or a serving loop whose
device memory is already owned by its own allocator.  w8_lmhead_argmax_noalloc
serves them with scratch kept inside the library.  Called through the C ABI,
it must give the same tokens and winning logits as w8_lmhead_argmax with a
workspace (bit for bit: same kernel, same arithmetic), on two calls in a row,
since every call reuses the scratch the previous one left behind.

This file is collected last on purpose, and also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verify_w4a16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _noalloc_fn(lib):
    fn = lib.w8_lmhead_argmax_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, I, I, I, P, P, P, P]
    fn.restype = I
    return fn


@pytest.mark.parametrize("M,K,V", [(16, 2560, 151936), (128, 256, 4096), (3, 128, 1000)])
def test_noalloc_matches_workspace_entry(w4v_mod, gpu, M, K, V):
    fn = _noalloc_fn(w4v_mod.load())
    X = torch.from_numpy(inputs.activations(21, M, K, "noalloc")).to(gpu)
    Wn, sn = inputs.lmhead_weights(21, V, K, "noalloc")
    W, s = torch.from_numpy(Wn).to(gpu), torch.from_numpy(sn).to(gpu)
    ref_max = torch.empty(M, dtype=torch.float32, device=gpu)
    ref = w4v_mod.w8_lmhead_argmax(X, W, s, maxlogit=ref_max)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        tok = torch.full((M,), -7, dtype=torch.int32, device=gpu)
        mx = torch.full((M,), float("nan"), dtype=torch.float32, device=gpu)
        code = fn(X.data_ptr(), W.data_ptr(), s.data_ptr(), M, K, V, tok.data_ptr(), mx.data_ptr(), None, stream)
        assert code == w4v_mod.OK, w4v_mod.status_string(code)
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), ref.cpu().numpy())
        assert np.array_equal(mx.cpu().numpy(), ref_max.cpu().numpy())
    assert w4v_mod.get_status() == w4v_mod.OK


def test_noalloc_rejects_rows_beyond_its_scratch(w4v_mod, gpu):
    fn = _noalloc_fn(w4v_mod.load())
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device=gpu)
    p = buf.data_ptr()
    code = fn(p, p, p, 129, 256, 1024, p, None, None, None)
    assert code == w4v_mod.ERR_SHAPE
