"""Pins for the oracle's verify GEMM: numpy's fp64 matmul (a library routine the
oracle does not call), the identity matrix (y = x bit for bit), an integer
closed form, and the bf16 bit-pattern decoding of known values."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (8, 40, 64), (33, 17, 130), (64, 96, 256)])
def test_gemm_matches_numpy_matmul(oracle_lib, M, N, K):
    x, w = synth.gemm_inputs(M * 1000 + N, M, N, K)
    y = oracle_lib.gemm(x, w)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(w).astype(np.float64).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_sampled_entries_match_full(oracle_lib):
    x, w = synth.gemm_inputs(3, 20, 30, 48)
    full = oracle_lib.gemm(x, w)
    s = np.array([[0, 0], [19, 29], [7, 11]], np.int32)
    y = oracle_lib.gemm(x, w, samples=s)
    assert np.array_equal(y, full[s[:, 0], s[:, 1]])


def _bf16_bits(values):
    """bf16 bit patterns of values that bf16 holds exactly (small integers)."""
    f = np.asarray(values, np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def test_gemm_identity_returns_x_exactly(oracle_lib):
    """W = I (bf16 1.0 on the diagonal): y is x itself, bit for bit."""
    M, K = 5, 48
    x, _ = synth.gemm_inputs(11, M, 1, K)
    w = np.zeros((K, K), np.uint16)
    w[np.arange(K), np.arange(K)] = 0x3F80
    y = oracle_lib.gemm(x, w)
    assert np.array_equal(y, synth.bf16_bits_to_f32(x).astype(np.float64))


def test_gemm_integer_closed_form(oracle_lib):
    """x[m][k] = m + 1 and w[n][k] = n - (k mod 3): y[m][n] = (m + 1) (K n - S)
    with S = sum_k (k mod 3), exact in fp64 (small integers)."""
    M, N, K = 6, 9, 30
    m, n, k = np.arange(M), np.arange(N), np.arange(K)
    x = _bf16_bits(np.broadcast_to((m + 1)[:, None], (M, K)))
    w = _bf16_bits(n[:, None] - (k % 3)[None, :])
    y = oracle_lib.gemm(x, w)
    S = int((k % 3).sum())
    expect = (m + 1)[:, None] * (K * n[None, :] - S)
    assert np.array_equal(y, expect.astype(np.float64))


def test_gemm_bf16_decoding(oracle_lib):
    """The bf16 inputs are decoded by their bit layout: 1 x 1 products of
    known patterns (1.0, -2.0, 0.5, the smallest normal, a subnormal)."""
    pats = np.array([0x3F80, 0xC000, 0x3F00, 0x0080, 0x0001], np.uint16)
    vals = [1.0, -2.0, 0.5, 2.0 ** -126, 2.0 ** -133]
    one = np.array([[0x3F80]], np.uint16)
    for p, v in zip(pats, vals):
        y = oracle_lib.gemm(np.array([[p]], np.uint16), one)
        assert y[0, 0] == v
