"""The oracle's pins reject plausible mistakes in the oracle itself.

Each case plants one mistake in a copy of oracle/oracle.c (a flipped sign, a
transposed operand, a wrong index or tie-break, a dropped term or factor),
compiles the copy on the CPU with gcc and runs the oracle's pin tests against
it in a child process: at least one pin has to fail.  The unmodified copy,
compiled and run the same way, passes them, so a failure is the planted
mistake's doing.  Every planted mistake keeps its accesses inside the buffers
the unmodified code touches.

The pins are the unit tests of the oracle (golden cases, closed forms,
brute force, invariants): tests/test_oracle_{gemm,lmhead,accept,ngram,gdn}.py.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

from conftest import ORACLE_UNDER_TEST, ROOT

SRC = os.path.join(ROOT, "oracle", "oracle.c")
GEMM, LMHEAD, ACCEPT, NGRAM, GDN = ("tests/test_oracle_%s.py" % n for n in ("gemm", "lmhead", "accept", "ngram", "gdn"))

# (name, function the mistake goes into, text replaced, replacement, pin files)
MUTANTS = [
    ("fp16 subnormal scale", "oracle_half_to_double",
     "ldexp((double)f, -24)", "ldexp((double)f, -25)", [GEMM]),
    ("fp16 exponent bias", "oracle_half_to_double",
     "e - 25)", "e - 24)", [GEMM]),
    ("zero point subtracted the wrong way", "oracle_dequant_w4",
     "((double)q[(size_t)n * K + k] - zero)", "(zero - (double)q[(size_t)n * K + k])", [GEMM]),
    ("default zero point 7", "oracle_dequant_w4",
     ": 8.0;", ": 7.0;", [GEMM]),
    ("scale table read [N][K/G]", "oracle_dequant_w4",
     "s[(size_t)g * N + n]", "s[(size_t)n * (K / G) + g]", [GEMM]),
    ("zero table read [N][K/G]", "oracle_dequant_w4",
     "z[(size_t)g * N + n]", "z[(size_t)n * (K / G) + g]", [GEMM]),
    ("groups in reverse order", "oracle_dequant_w4",
     "int g = k / G;", "int g = (K - 1 - k) / G;", [GEMM]),
    ("weights not transposed", "oracle_matmul_dequantized",
     "w[(size_t)n * K + k]", "w[(size_t)k * N + n]", [GEMM]),
    ("first product term dropped", "oracle_matmul_dequantized",
     "for (int k = 0; k < K; ++k) acc", "for (int k = 1; k < K; ++k) acc", [GEMM]),
    ("sampled: zero point subtracted the wrong way", "oracle_w4a16_gemm_sampled",
     "((double)q[(size_t)n * K + k] - zero)", "(zero - (double)q[(size_t)n * K + k])", [GEMM]),
    ("sampled: scale table read [N][K/G]", "oracle_w4a16_gemm_sampled",
     "s[(size_t)g * N + n]", "s[(size_t)n * (K / G) + g]", [GEMM]),
    ("lm_head row scale dropped", "oracle_lmhead_logits",
     "= scale * acc;", "= acc;", [LMHEAD]),
    ("lm_head weights not transposed", "oracle_lmhead_logits",
     "W[(size_t)v * K + k]", "W[(size_t)k * V + v]", [LMHEAD]),
    ("lm_head rows: row scale dropped", "oracle_lmhead_argmax_rows",
     "double l = oracle_half_to_double(s[v]) * acc;", "double l = acc;", [LMHEAD]),
    ("lm_head rows: ties to the last index", "oracle_lmhead_argmax_rows",
     "else if (l > b1)", "else if (l >= b1)", [LMHEAD]),
    ("lm_head rows: second best not kept", "oracle_lmhead_argmax_rows",
     "else if (l > b2) b2 = l;", "", [LMHEAD]),
    ("argmax ties to the last index", "oracle_argmax_f64",
     "if (x > best)", "if (x >= best)", [LMHEAD]),
    ("fp32 argmax ties to the last index", "oracle_argmax_f32",
     "if (x > best)", "if (x >= best)", [LMHEAD]),
    ("draft compared with the next target", "oracle_spec_accept",
     "db[n] == tb[n])", "db[n] == tb[n + 1])", [ACCEPT]),
    ("bonus token counted as accepted", "oracle_spec_accept",
     "n_out[b] = n;", "n_out[b] = n + 1;", [ACCEPT]),
    ("emitted slots past the bonus token not -1", "oracle_spec_accept",
     "tb[n] : -1)", "tb[n] : tb[n])", [ACCEPT]),
    ("earliest occurrence instead of the latest", "oracle_ngram_draft",
     "for (int p = L - n - 1; p >= 0; --p)", "for (int p = 0; p <= L - n - 1; ++p)", [NGRAM]),
    ("shortest n-gram first", "oracle_ngram_draft",
     "for (int n = n_max; n >= n_min && found_n == 0; --n)",
     "for (int n = n_min; n <= n_max && found_n == 0; ++n)", [NGRAM]),
    ("continuation starts one token early", "oracle_ngram_draft",
     "d[i] = c[p + n + i];", "d[i] = c[p + n + i - 1];", [NGRAM]),
    ("n-gram may overlap its own position", "oracle_ngram_draft",
     "for (int p = L - n - 1;", "for (int p = L - n;", [NGRAM]),
    ("erase term added instead of subtracted", "oracle_gdn_recurrence",
     "(m == j ? 1.0 : 0.0) - beta[t]", "(m == j ? 1.0 : 0.0) + beta[t]", [GDN]),
    ("decay applied to the new write too", "oracle_gdn_recurrence",
     "alpha[t] * P[(size_t)i * dk + j] + beta[t] * vt[i] * kt[j];",
     "alpha[t] * (P[(size_t)i * dk + j] + beta[t] * vt[i] * kt[j]);", [GDN]),
    ("write strength dropped from the write", "oracle_gdn_recurrence",
     "+ beta[t] * vt[i] * kt[j];", "+ vt[i] * kt[j];", [GDN]),
    ("output read before the write", "oracle_gdn_recurrence",
     "acc += S[(size_t)i * dk + j] * qt[j];", "acc += P[(size_t)i * dk + j] * qt[j];", [GDN]),
]


def _function_span(src, name):
    """[start, end) of the C function `name`: from its signature to the first
    closing brace at column 0 after it."""
    start = src.index("\n" + _signature_prefix(src, name))
    end = src.index("\n}\n", start) + 3
    return start, end


def _signature_prefix(src, name):
    for kind in ("void ", "double ", "int "):
        if ("\n" + kind + name + "(") in src:
            return kind + name + "("
    raise AssertionError("no function %s in oracle.c" % name)


def _plant(src, func, old, new):
    a, b = _function_span(src, func)
    body = src[a:b]
    assert body.count(old) == 1, "the text to replace must occur exactly once in %s: %r" % (func, old)
    return src[:a] + body.replace(old, new) + src[b:]


def _run_pins(tmp, tag, source, files):
    """Compile `source` as a shared library and run the pin files against it;
    returns (exit code, last lines of the output)."""
    c_path = os.path.join(tmp, tag + ".c")
    so_path = os.path.join(tmp, tag + ".so")
    with open(c_path, "w") as f:
        f.write(source)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", c_path, "-o", so_path, "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, **{ORACLE_UNDER_TEST: so_path})
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, "\n".join((r.stdout + r.stderr).strip().splitlines()[-3:])


@pytest.fixture(scope="module")
def outcomes(oracle_mod, tmp_path_factory):
    """Every mutant and the unmodified control, run in parallel child processes."""
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    with open(SRC) as f:
        src = f.read()
    jobs = {"control": (src, sorted({f for m in MUTANTS for f in m[4]}))}
    for i, (name, func, old, new, files) in enumerate(MUTANTS):
        jobs[name] = (_plant(src, func, old, new), files)
    with cf.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futs = {name: ex.submit(_run_pins, tmp, "m%02d" % i, s, files)
                for i, (name, (s, files)) in enumerate(jobs.items())}
        return {name: fut.result() for name, fut in futs.items()}


def test_unmodified_copy_passes_the_pins(outcomes):
    code, tail = outcomes["control"]
    assert code == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(outcomes, name):
    code, tail = outcomes[name]
    assert code == 1 and "failed" in tail, "the pins did not catch: %s\n%s" % (name, tail)
