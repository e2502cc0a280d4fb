"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/w4v.h declares, packs int4 weights in the documented
layout, sizes workspaces, and rejects bad arguments before launching
anything.  Every call here with fake pointers fails validation, so nothing
ever reaches a kernel."""
import ctypes

import numpy as np
import pytest

FAKE = 0x10000          # an aligned, never-dereferenced stand-in pointer


def test_exports_every_header_function(w4v_mod):
    names = w4v_mod.header_functions()
    for required in ("w4v_init", "w4v_get_status", "w4v_pack_int4", "w4a16_gemm",
                     "w8_lmhead_argmax", "spec_accept", "w8_lmhead_argmax_accept", "ngram_draft",
                     "gdn_verify", "gdn_commit", "gdn_step"):
        assert required in names
    lib = w4v_mod.load()
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(w4v_mod):
    for code in range(8):
        s = w4v_mod.status_string(code)
        assert isinstance(s, str) and s
    assert w4v_mod.status_string(0) == "ok"
    assert w4v_mod.status_string(99) == "unknown status"


@pytest.mark.parametrize("N,K", [(128, 128), (512, 256), (200, 384), (8, 128), (7680, 2560)])
def test_pack_roundtrip(w4v_mod, N, K):
    q = np.random.default_rng(N + K).integers(0, 16, size=(N, K), dtype=np.uint8)
    packed = w4v_mod.pack_int4(q)
    assert packed.size == -(-N // 128) * 128 * K // 2
    assert np.array_equal(w4v_mod.unpack_int4(packed, N, K), q)


def test_pack_layout_documented(w4v_mod):
    """Spot-check the header's description: block (tile, group) is 8192 bytes,
    chunk j of row r at (j*128 + r)*16, word w covers k = 32j+8w..+7, nibble i
    holds k offset {0,2,4,6,1,3,5,7}[i]."""
    N, K = 256, 256
    q = np.random.default_rng(1).integers(0, 16, size=(N, K), dtype=np.uint8)
    packed = w4v_mod.pack_int4(q)
    order = [0, 2, 4, 6, 1, 3, 5, 7]
    rng = np.random.default_rng(2)
    for _ in range(200):
        n, k = int(rng.integers(0, N)), int(rng.integers(0, K))
        t, r, g = n // 128, n % 128, k // 128
        kk = k % 128
        j, w, off = kk // 32, (kk % 32) // 8, kk % 8
        i = order.index(off)
        base = (t * (K // 128) + g) * 8192 + (j * 128 + r) * 16 + 4 * w
        word = int.from_bytes(packed[base:base + 4].tobytes(), "little")
        assert (word >> (4 * i)) & 15 == q[n, k]


def test_pack_pads_tail_rows_with_zero_point(w4v_mod):
    N, K = 136, 128
    q = np.zeros((N, K), np.uint8)
    packed = w4v_mod.pack_int4(q)
    tail = packed[8192:].reshape(4, 128, 16)[:, 8:, :]     # rows 136.. of the second tile
    assert np.all(tail == 0x88)


def test_workspace_sizes(w4v_mod):
    assert w4v_mod.w4a16_workspace_bytes(16, 7680, 2560) > 0
    assert w4v_mod.w4a16_workspace_bytes(33, 512, 256) >= 256 * 128 * 4   # prefill: split-tile partials
    assert w4v_mod.w4a16_workspace_bytes(-1, 512, 256) == 0
    assert w4v_mod.w4a16_workspace_bytes(16, 100, 256) == 0       # N % 8 != 0
    assert w4v_mod.w8_lmhead_argmax_workspace_bytes(128, 151936) > 0
    assert w4v_mod.w8_lmhead_argmax_workspace_bytes(129, 151936) == 0
    assert w4v_mod.packed_bytes(100, 256) == 0


def test_argument_validation_before_launch(w4v_mod):
    lib = w4v_mod.load()
    ws_small = 16
    # w4a16_gemm
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 64, FAKE, 16, 512, 256, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    # group size 32 passes the shape checks (and fails later on the workspace)
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 32, FAKE, 16, 512, 256, FAKE, ws_small, None) == w4v_mod.ERR_WORKSPACE
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 128, FAKE, -1, 512, 256, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 128, FAKE, 16, 500, 256, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 128, FAKE, 16, 512, 200, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, FAKE, 128, FAKE, 16, 520, 256, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w4a16_gemm(None, FAKE, FAKE, None, 128, FAKE, 16, 512, 256, FAKE, 1 << 30, None) == w4v_mod.ERR_ARG
    assert lib.w4a16_gemm(FAKE + 2, FAKE, FAKE, None, 128, FAKE, 16, 512, 256, FAKE, 1 << 30, None) == w4v_mod.ERR_ALIGN
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 128, FAKE, 16, 512, 256, FAKE, ws_small, None) == w4v_mod.ERR_WORKSPACE
    assert lib.w4a16_gemm(FAKE, FAKE, FAKE, None, 128, FAKE, 16, 512, 256, None, 1 << 30, None) == w4v_mod.ERR_WORKSPACE
    assert lib.w4a16_gemm(None, None, None, None, 128, None, 0, 512, 256, None, 0, None) == w4v_mod.OK   # M == 0
    # w4a16_gemm_ex: the same checks plus unknown flag bits
    assert lib.w4a16_gemm_ex(FAKE, FAKE, FAKE, None, 128, FAKE, 16, 512, 256, FAKE, 1 << 30, 4, None) == w4v_mod.ERR_ARG
    # the batch-invariant path for M > 32 needs the 32-row workspace as well
    assert w4v_mod.w4a16_workspace_bytes(128, 2560, 2560) >= w4v_mod.w4a16_workspace_bytes(32, 2560, 2560)
    assert lib.w4a16_gemm_ex(FAKE, FAKE, FAKE, None, 128, FAKE, 128, 512, 256, FAKE, 1 << 20, 3, None) == w4v_mod.ERR_WORKSPACE
    assert lib.w4a16_gemm_ex(FAKE, FAKE, FAKE, None, 128, FAKE, 16, 500, 256, FAKE, 1 << 30, 1, None) == w4v_mod.ERR_SHAPE
    assert lib.w4a16_gemm_ex(None, None, None, None, 128, None, 0, 512, 256, None, 0, 1, None) == w4v_mod.OK
    # w8_lmhead_argmax
    assert lib.w8_lmhead_argmax(FAKE, FAKE, FAKE, 129, 256, 1024, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w8_lmhead_argmax(FAKE, FAKE, FAKE, 16, 200, 1024, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w8_lmhead_argmax(FAKE, FAKE, FAKE, 16, 256, 1020, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert lib.w8_lmhead_argmax(FAKE, FAKE, None, 16, 256, 1024, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ARG
    assert lib.w8_lmhead_argmax(FAKE, FAKE + 8, FAKE, 16, 256, 1024, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ALIGN
    assert lib.w8_lmhead_argmax(FAKE, FAKE, FAKE, 16, 256, 1024, FAKE, None, None, FAKE, ws_small, None) == w4v_mod.ERR_WORKSPACE
    assert lib.w8_lmhead_argmax(None, None, None, 0, 256, 1024, None, None, None, None, 0, None) == w4v_mod.OK
    # w8_lmhead_argmax_ex / _accept_ex: unknown flag bits, then the same checks
    ex = lib.w8_lmhead_argmax_ex
    assert ex(FAKE, FAKE, FAKE, 16, 256, 1024, FAKE, None, None, FAKE, 1 << 30, 1, None) == w4v_mod.ERR_ARG
    assert ex(FAKE, FAKE, FAKE, 129, 256, 1024, FAKE, None, None, FAKE, 1 << 30, 2, None) == w4v_mod.ERR_SHAPE
    assert ex(FAKE, FAKE, FAKE, 64, 256, 1024, FAKE, None, None, FAKE, ws_small, 2, None) == w4v_mod.ERR_WORKSPACE
    assert ex(None, None, None, 0, 256, 1024, None, None, None, None, 0, 2, None) == w4v_mod.OK
    aex = lib.w8_lmhead_argmax_accept_ex
    assert aex(FAKE, FAKE, FAKE, 8, 15, 256, 1024, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, 4,
               None) == w4v_mod.ERR_ARG
    assert aex(FAKE, FAKE, FAKE, 8, 16, 256, 1024, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, 2,
               None) == w4v_mod.ERR_SHAPE
    assert aex(None, None, None, 0, 15, 256, 1024, None, None, None, None, None, None, 0, 2, None) == w4v_mod.OK
    # spec_accept
    assert lib.spec_accept(FAKE, FAKE, 4, 1025, FAKE, None, None) == w4v_mod.ERR_SHAPE
    assert lib.spec_accept(FAKE, FAKE, -1, 4, FAKE, None, None) == w4v_mod.ERR_SHAPE
    assert lib.spec_accept(None, FAKE, 4, 4, FAKE, None, None) == w4v_mod.ERR_ARG
    assert lib.spec_accept(FAKE, None, 4, 4, FAKE, None, None) == w4v_mod.ERR_ARG
    assert lib.spec_accept(FAKE + 1, FAKE, 4, 4, FAKE, None, None) == w4v_mod.ERR_ALIGN
    assert lib.spec_accept(None, None, 0, 4, None, None, None) == w4v_mod.OK
    # w8_lmhead_argmax_accept: B*(n_draft+1) rows, at most 128
    acc = lib.w8_lmhead_argmax_accept
    assert acc(FAKE, FAKE, FAKE, 8, 16, 256, 1024, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert acc(FAKE, FAKE, FAKE, 129, 0, 256, 1024, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert acc(FAKE, FAKE, FAKE, 1, -1, 256, 1024, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert acc(FAKE, FAKE, FAKE, 1, 15, 200, 1024, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert acc(FAKE, FAKE, FAKE, 1, 15, 256, 1024, None, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ARG
    assert acc(FAKE, FAKE, FAKE, 1, 15, 256, 1024, FAKE, FAKE, None, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ARG
    assert acc(FAKE, FAKE, FAKE, 1, 15, 256, 1024, FAKE + 2, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ALIGN
    assert acc(FAKE, FAKE, FAKE, 1, 15, 256, 1024, FAKE, FAKE, FAKE, None, None, FAKE, ws_small, None) == w4v_mod.ERR_WORKSPACE
    assert acc(None, None, None, 0, 15, 256, 1024, None, None, None, None, None, None, 0, None) == w4v_mod.OK
    # ngram_draft
    ng = lib.ngram_draft
    assert ng(FAKE, FAKE, 4, 100, 0, 3, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE   # n_min 0
    assert ng(FAKE, FAKE, 4, 100, 3, 2, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE   # n_max < n_min
    assert ng(FAKE, FAKE, 4, 100, 1, 65, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert ng(FAKE, FAKE, 4, 100, 1, 3, 1025, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert ng(FAKE, FAKE, 4, 0, 1, 3, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE     # ld 0
    assert ng(FAKE, FAKE, 65536, 100, 1, 3, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_SHAPE
    assert ng(None, FAKE, 4, 100, 1, 3, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ARG
    assert ng(FAKE, FAKE, 4, 100, 1, 3, 8, None, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ARG
    assert ng(FAKE, FAKE + 2, 4, 100, 1, 3, 8, FAKE, None, FAKE, 1 << 30, None) == w4v_mod.ERR_ALIGN
    assert ng(FAKE, FAKE, 4, 100, 1, 3, 8, FAKE, None, FAKE, 16, None) == w4v_mod.ERR_WORKSPACE
    assert ng(None, None, 0, 100, 1, 3, 8, None, None, None, 0, None) == w4v_mod.OK
    assert w4v_mod.load().ngram_draft_workspace_bytes(8) >= 8 * 12
    # gdn_verify / gdn_commit
    gv, gc = lib.gdn_verify, lib.gdn_commit
    assert gv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 16, 4, 64, 128, FAKE, None) == w4v_mod.ERR_SHAPE    # dk != 128
    assert gv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 65, 4, 128, 128, FAKE, None) == w4v_mod.ERR_SHAPE   # T > 64
    assert gv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 4, 128, 128, FAKE, None) == w4v_mod.ERR_SHAPE
    assert gv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 16, 4, 128, 100, FAKE, None) == w4v_mod.ERR_SHAPE   # dv % 32
    assert gv(FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 16, 4, 128, 128, FAKE, None) == w4v_mod.ERR_ARG
    assert gv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 16, 4, 128, 128, None, None) == w4v_mod.ERR_ARG
    assert gv(FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 16, 4, 128, 128, FAKE, None) == w4v_mod.ERR_ALIGN
    assert gv(None, None, None, None, None, None, 0, 16, 4, 128, 128, None, None) == w4v_mod.OK
    assert gc(FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 16, 4, 128, 128, None) == w4v_mod.ERR_ARG
    assert gc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 1, 16, 4, 128, 128, None) == w4v_mod.ERR_ALIGN
    assert gc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 16, 0, 128, 128, None) == w4v_mod.ERR_SHAPE
    # gdn_step(state, k_prev, v_prev, alpha_prev, beta_prev, n_prev, T_prev, q, k, v, alpha, beta,
    #          B, T, H, dk, dv, o, stream)
    gs = lib.gdn_step
    F = FAKE
    assert gs(F, F, F, F, F, F, 65, F, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_SHAPE   # T_prev > 64
    assert gs(F, F, F, F, F, F, -1, F, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_SHAPE
    assert gs(F, F, F, F, F, F, 16, F, F, F, F, F, 1, 65, 4, 128, 128, F, None) == w4v_mod.ERR_SHAPE   # T > 64
    assert gs(F, F, F, F, F, None, 16, F, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_ARG  # no n_prev
    assert gs(F, None, F, F, F, F, 16, F, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_ARG  # no k_prev
    assert gs(F, F, F, F, F, F + 2, 16, F, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_ALIGN
    assert gs(F, F + 4, F, F, F, F, 16, F, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_ALIGN
    assert gs(F, F, F, F, F, F, 16, None, F, F, F, F, 1, 16, 4, 128, 128, F, None) == w4v_mod.ERR_ARG  # no q
    assert gs(F, F, F, F, F, F, 16, F, F, F, F, F, 1, 16, 4, 128, 128, None, None) == w4v_mod.ERR_ARG  # no o
    assert gs(None, None, None, None, None, None, 0, None, None, None, None, None, 0, 16, 4, 128, 128, None,
              None) == w4v_mod.OK
    # packer
    assert lib.w4v_pack_int4(None, 128, 128, FAKE) == w4v_mod.ERR_ARG
    buf = ctypes.create_string_buffer(16)
    assert lib.w4v_pack_int4(ctypes.addressof(buf), 100, 128, ctypes.addressof(buf)) == w4v_mod.ERR_SHAPE


def test_grouped_argument_validation_before_launch(w4v_mod):
    """w4a16_grouped_plan / w4a16_gemm_grouped reject bad arguments before any
    device work: sizes, null or misaligned pointers, mixed zero tables, a
    small or misaligned plan, unknown flags and handles not written by the
    planner."""
    lib = w4v_mod.load()
    Pr = w4v_mod.Problem

    def probs(*specs):
        arr = (Pr * len(specs))()
        for i, (A, Bq, sc, z, C, N, K) in enumerate(specs):
            arr[i] = Pr(A, Bq, sc, z, C, N, K)
        return arr

    F = FAKE
    good = (F, F, F, None, F, 512, 256)
    big = 1 << 30
    h = w4v_mod.GroupedHandle()
    plan = lib.w4a16_grouped_plan
    hb = ctypes.byref(h)
    assert lib.w4a16_grouped_plan_bytes(0) == 0
    assert lib.w4a16_grouped_plan_bytes(4097) == 0
    assert lib.w4a16_grouped_plan_bytes(4) >= 4 * 3 * 128
    assert plan(probs(good), 0, 16, 128, F, big, hb, None) == w4v_mod.ERR_SHAPE          # no problem
    assert plan(probs(good), 4097, 16, 128, F, big, hb, None) == w4v_mod.ERR_SHAPE
    assert plan(probs(good), 1, 0, 128, F, big, hb, None) == w4v_mod.ERR_SHAPE           # M = 0
    assert plan(probs(good), 1, 33, 128, F, big, hb, None) == w4v_mod.ERR_SHAPE          # M > 32
    assert plan(probs(good), 1, 16, 64, F, big, hb, None) == w4v_mod.ERR_SHAPE           # group
    assert plan(None, 1, 16, 128, F, big, hb, None) == w4v_mod.ERR_ARG
    assert plan(probs(good), 1, 16, 128, None, big, hb, None) == w4v_mod.ERR_ARG
    assert plan(probs(good), 1, 16, 128, F, big, None, None) == w4v_mod.ERR_ARG
    assert plan(probs((F, F, F, None, F, 500, 256)), 1, 16, 128, F, big, hb, None) == w4v_mod.ERR_SHAPE
    assert plan(probs((F, F, F, None, F, 512, 200)), 1, 16, 128, F, big, hb, None) == w4v_mod.ERR_SHAPE
    assert plan(probs((F, F, F, F, F, 512, 256), (F, F, F, F, F, 520, 256)), 2, 16, 128, F, big, hb,
                None) == w4v_mod.ERR_SHAPE                                                    # zeros: N % 16
    assert plan(probs(good, (F, F, F, F, F, 512, 256)), 2, 16, 128, F, big, hb, None) == w4v_mod.ERR_ARG
    assert plan(probs(good, (F, F, None, None, F, 512, 256)), 2, 16, 128, F, big, hb, None) == w4v_mod.ERR_ARG
    assert plan(probs(good, (F, F + 8, F, None, F, 512, 256)), 2, 16, 128, F, big, hb, None) == w4v_mod.ERR_ALIGN
    assert plan(probs(good, (F, F, F, None, F + 2, 512, 256)), 2, 16, 128, F, big, hb, None) == w4v_mod.ERR_ALIGN
    assert plan(probs(good), 1, 16, 128, F, 16, hb, None) == w4v_mod.ERR_WORKSPACE      # plan too small
    assert plan(probs(good), 1, 16, 128, F + 16, big, hb, None) == w4v_mod.ERR_ALIGN    # plan not 64-aligned
    # a handle the planner did not write (or changed since) is refused
    assert lib.w4a16_grouped_workspace_bytes(hb) == 0
    assert lib.w4a16_grouped_workspace_bytes(None) == 0
    assert lib.w4a16_gemm_grouped(hb, F, big, 0, None) == w4v_mod.ERR_ARG
    assert lib.w4a16_gemm_grouped(None, F, big, 0, None) == w4v_mod.ERR_ARG
    h.plan, h.units, h.n_problems, h.M, h.group, h.tiles = F, 10, 1, 16, 128, 1
    assert lib.w4a16_gemm_grouped(hb, F, big, 0, None) == w4v_mod.ERR_ARG
    assert lib.w4a16_gemm_grouped(hb, F, big, 2, None) == w4v_mod.ERR_ARG             # unknown flag


def test_split_owner_matches_even_split():
    """Host restatement check of the stream-K ownership formula used by the kernels:
    owner(u) = ((u+1)P - 1) // U is the CTA whose [cU/P, (c+1)U/P) holds u."""
    for U in (1, 7, 10, 400, 1200, 1520, 3040):
        for P in (1, 3, 4, 148, 152):
            if P > U:
                continue
            for c in range(P):
                lo, hi = c * U // P, (c + 1) * U // P
                assert hi > lo
                for u in (lo, hi - 1):
                    assert ((u + 1) * P - 1) // U == c
