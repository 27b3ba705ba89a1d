"""Pin for the oracle's verify GEMM: numpy's fp64 matmul (a library routine)."""
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
