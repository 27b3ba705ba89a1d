"""C-ABI checks that need no GPU: the library loads, exports every entry
point the header declares, and rejects invalid arguments on the host before
anything is enqueued (so none of these calls touches a device)."""
import ctypes
import os
import re

import numpy as np
import pytest

import speculative_decoding_verification_attention_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    return sv.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    assert set(names) == set(sv.EXPORTED_SYMBOLS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert lib.spec_status_string(0) == b"SPEC_OK"
    assert lib.spec_status_string(3) == b"SPEC_ERR_WORKSPACE"
    assert lib.spec_status_string(99) == b"SPEC_ERR_UNKNOWN"
    assert lib.spec_version() >= 100


P = ctypes.c_void_p
FAKE = P(0x7F0000001000)   # never dereferenced: validation fails first


def test_accept_greedy_rejects_bad_arguments(lib):
    f = lib.spec_accept_greedy
    assert f(FAKE, FAKE, -1, 3, 10, FAKE, FAKE, None, None) == INVALID
    assert f(FAKE, FAKE, 1, -1, 10, FAKE, FAKE, None, None) == INVALID
    assert f(FAKE, FAKE, 1, 3, 0, FAKE, FAKE, None, None) == INVALID
    assert f(FAKE, FAKE, 1, 64, 10, FAKE, FAKE, None, None) == UNSUPPORTED
    assert f(None, FAKE, 1, 3, 10, FAKE, FAKE, None, None) == INVALID
    assert f(FAKE, None, 1, 3, 10, FAKE, FAKE, None, None) == INVALID
    assert f(P(0x7F0000001002), FAKE, 1, 3, 10, FAKE, FAKE, None, None) == INVALID
    assert f(None, None, 0, 3, 10, None, None, None, None) == 0   # empty batch: no-op


def test_accept_sample_rejects_bad_arguments(lib):
    f = lib.spec_accept_sample
    W = 1 << 20
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 3, 0, FAKE, FAKE, FAKE, W, None, None) == INVALID
    assert f(FAKE, None, FAKE, FAKE, FAKE, 1, 3, 10, FAKE, FAKE, FAKE, W, None, None) == INVALID
    assert f(FAKE, FAKE, FAKE, None, FAKE, 1, 3, 10, FAKE, FAKE, FAKE, W, None, None) == INVALID
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 3, 10, FAKE, FAKE, FAKE, W, None, None) == INVALID
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 70, 10, FAKE, FAKE, FAKE, W, None, None) == UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 3, 10, FAKE, FAKE, None, W, None, None) == WORKSPACE
    need = lib.spec_accept_sample_workspace_size(4, 1000)
    assert need > 0
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 3, 1000, FAKE, FAKE, FAKE, need - 1, None, None) == WORKSPACE
    assert f(None, None, None, None, None, 0, 3, 10, None, None, None, 0, None, None) == 0


def test_gemm_rejects_bad_arguments(lib):
    f = lib.spec_verify_gemm
    assert f(FAKE, FAKE, FAKE, -1, 128, 64, None, 0, None, None) == INVALID
    assert f(FAKE, FAKE, FAKE, 8, 100, 64, None, 0, None, None) == UNSUPPORTED   # N % 128
    assert f(FAKE, FAKE, FAKE, 8, 128, 60, None, 0, None, None) == UNSUPPORTED   # K % 64
    assert f(None, FAKE, FAKE, 8, 128, 64, None, 0, None, None) == INVALID
    assert f(P(0x7F0000001008), FAKE, FAKE, 8, 128, 64, None, 0, None, None) == INVALID
    assert f(None, None, None, 0, 128, 64, None, 0, None, None) == 0   # empty: no-op
    # weight streaming: 4 KB of arrival counters, then fp32 partial tiles as
    # wide as the padded x rows, two per CTA
    ws8 = lib.spec_verify_gemm_workspace_size(8, 6144, 6144)
    assert ws8 >= 4096 + 2 * 128 * 32 * 4 and ws8 % 256 == 0
    assert ws8 < lib.spec_verify_gemm_workspace_size(256, 6144, 6144)
    # pairs of CTAs on whole tiles: no workspace
    assert lib.spec_verify_gemm_workspace_size(512, 6144, 6144) == 0
    assert lib.spec_verify_gemm_workspace_size(257, 6144, 6144) == 0


def test_tree_entry_points_reject_bad_arguments(lib):
    f = lib.spec_verify_tree_attention
    W = 1 << 30
    args = lambda parent, D=3: (FAKE, FAKE, FAKE, 10, FAKE, 4, FAKE, parent, 2, D, 1, 4, 64, 16, 0.125,
                                FAKE, None, FAKE, W, None, None)
    assert f(*args(None)) == INVALID                       # a tree needs its parents
    assert f(*args(P(0x7F0000001002))) == INVALID          # misaligned parents
    assert f(*args(FAKE, D=64)) == UNSUPPORTED             # at most 64 nodes
    chain = lib.spec_verify_attention_workspace_size(2, 3, 1, 4, 64, 64)
    tree = lib.spec_verify_tree_attention_workspace_size(2, 3, 1, 4, 64, 64)
    assert tree >= chain + 2 * 4 * 8
    g = lib.spec_accept_tree_greedy
    assert g(FAKE, FAKE, None, 2, 3, 10, FAKE, FAKE, None, None, None) == INVALID
    assert g(FAKE, None, FAKE, 2, 3, 10, FAKE, FAKE, None, None, None) == INVALID
    assert g(FAKE, FAKE, FAKE, 2, 64, 10, FAKE, FAKE, None, None, None) == UNSUPPORTED
    assert g(FAKE, FAKE, FAKE, 2, 3, 0, FAKE, FAKE, None, None, None) == INVALID
    assert g(None, None, None, 0, 3, 10, None, None, None, None, None) == 0
    h = lib.spec_accept_tree_sample
    args = lambda q=FAKE, ua=FAKE, D=3, V=10, B=2: (FAKE, q, FAKE, FAKE, ua, FAKE, B, D, V, FAKE, FAKE, None,
                                                    None, None)
    assert h(*args(q=None)) == INVALID                      # the draft rows are needed
    assert h(*args(ua=None)) == INVALID
    assert h(*args(ua=P(0x7F0000001002))) == INVALID        # misaligned uniforms
    assert h(*args(D=64)) == UNSUPPORTED
    assert h(*args(V=(1 << 22) + 1)) == UNSUPPORTED
    assert h(*args(V=0)) == INVALID
    assert h(None, None, None, None, None, None, 0, 3, 10, None, None, None, None, None) == 0


def test_logits_acceptance_rejects_bad_arguments(lib):
    f = lib.spec_accept_sample_logits
    W = 1 << 30
    args = lambda T=1.0, zp=FAKE, zq=FAKE, dr=FAKE, B=2, D=3, V=10, ws=FAKE, wb=W: (
        zp, zq, dr, T, 7, B, D, V, FAKE, FAKE, ws, wb, None, None)
    assert f(*args(T=0.0)) == INVALID
    assert f(*args(T=-1.0)) == INVALID
    assert f(*args(T=float("nan"))) == INVALID
    assert f(*args(T=float("inf"))) == INVALID
    assert f(*args(zp=None)) == INVALID
    assert f(*args(zq=None)) == INVALID
    assert f(*args(dr=None)) == INVALID
    assert f(*args(zp=P(0x7F0000001002))) == INVALID
    assert f(*args(V=0)) == INVALID
    assert f(*args(D=64)) == UNSUPPORTED
    assert f(*args(ws=None)) == WORKSPACE
    need = lib.spec_accept_sample_logits_workspace_size(2, 3, 10)
    assert need >= lib.spec_accept_sample_workspace_size(2, 10) + 2 * 7 * 8
    assert f(*args(wb=need - 1)) == WORKSPACE
    assert f(*args(zq=None, dr=None, D=0, B=0)) == 0   # empty batch: no-op
    assert lib.spec_accept_sample_logits_workspace_size(2, 64, 10) == 0


def test_adasd_rejects_bad_arguments(lib):
    f = lib.spec_accept_adasd
    W = 1 << 30
    args = lambda th=1.0, tj=0.2, p=FAKE, q=FAKE, dr=FAKE, ua=FAKE, B=2, D=3, V=10, ws=FAKE, wb=W: (
        p, q, dr, ua, FAKE, th, tj, B, D, V, FAKE, FAKE, None, None, None, ws, wb, None, None)
    assert f(*args(th=float("nan"))) == INVALID
    assert f(*args(tj=float("nan"))) == INVALID
    assert f(*args(p=None)) == INVALID
    assert f(*args(q=None)) == INVALID
    assert f(*args(dr=None)) == INVALID
    assert f(*args(ua=None)) == INVALID
    assert f(*args(p=P(0x7F0000001002))) == INVALID
    assert f(*args(D=64)) == UNSUPPORTED
    assert f(*args(ws=None)) == WORKSPACE
    need = lib.spec_accept_adasd_workspace_size(2, 3, 10)
    assert need >= lib.spec_accept_sample_workspace_size(2, 10) + 2 * 3 * 8
    assert f(*args(wb=need - 1)) == WORKSPACE
    assert f(*args(q=None, dr=None, ua=None, D=0, B=0)) == 0   # empty batch: no-op
    assert f(*args(th=float("inf"), tj=float("-inf"), B=0)) == 0


def test_selftest_bounded_wait_rejects_bad_arguments(lib):
    f = lib.spec_selftest_bounded_wait
    never = 0xFFFFFFFFFFFFFFFF
    assert f(0, never, FAKE, None, None) == INVALID                  # no limit
    assert f(10_000_000_001, never, FAKE, None, None) == INVALID     # limit above 10 s
    assert f(1_000_000, 10_000_000_001, FAKE, None, None) == INVALID  # arrival later than 10 s
    assert f(1_000_000, never, None, None, None) == INVALID          # no result buffer
    assert f(1_000_000, never, P(0x7F0000001004), None, None) == INVALID   # misaligned result
