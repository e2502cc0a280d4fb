"""The product path has no CPU fallback: without the library, or without a
GB300, calls raise instead of computing anything on the host."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_missing_library_raises():
    code = ("from speculative_decoding_verify_w4a16_gb300 import w4v\n"
            "w4v.load('/nonexistent/libw4v.so')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "not built" in r.stderr


def test_init_without_gb300_raises(w4v_mod):
    """On a machine without an sm_103 device the library reports an error
    (no kernel, no host computation)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(w4v_mod.W4VError) as e:
        w4v_mod.init()
    assert e.value.code in (w4v_mod.ERR_ARCH, w4v_mod.ERR_CUDA)
