"""The bounded device wait, made to run out on purpose.

Every mbarrier wait in the library's kernels gives up after a limit, records
SPEC_DEV_ERR_TIMEOUT in the caller's status word, stops the kernel's other
roles and returns, so that a stalled copy or a lost arrival never hangs the
GPU.  spec_selftest_bounded_wait runs that same wait in a one-CTA kernel on
a barrier that nothing arrives on (a flag that nothing sets), with no copy
or MMA in flight; the kernel must return, report the timeout, and leave the
context usable for the next call.
"""
import numpy as np
import pytest

import oracle
import synth

TIMEOUT_BIT = 0x4


@pytest.fixture(scope="module")
def sv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


@pytest.mark.gpu
def test_wait_that_runs_out_reports_timeout_and_returns(sv):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    limit = 2_000_000                                   # 2 ms
    res = sv.selftest_bounded_wait(limit, None, dev_status=st)
    torch.cuda.synchronize()
    done, abort, waited = res.cpu().tolist()
    assert done == 0 and abort == 1
    assert int(st.item()) & TIMEOUT_BIT
    assert limit <= waited < 1_000_000_000              # gave up after the limit, not much later


@pytest.mark.gpu
def test_wait_that_is_arrived_on_completes(sv):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = sv.selftest_bounded_wait(1_000_000_000, 200_000, dev_status=st)   # arrival after 0.2 ms
    torch.cuda.synchronize()
    done, abort, waited = res.cpu().tolist()
    assert done == 1 and abort == 0
    assert int(st.item()) == 0
    assert waited < 500_000_000


@pytest.mark.gpu
def test_context_usable_after_a_timeout(sv):
    """A verify-attention call right after an expired wait matches the oracle."""
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.selftest_bounded_wait(1_000_000, None, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & TIMEOUT_BIT
    D, Hkv, G, d = 3, 2, 4, 128
    inp = synth.attention_inputs(5, 2, Hkv, G, d, D, [300, 517], page_size=64)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sv.verify_attention(bf16(inp.q), bf16(inp.k_pages), bf16(inp.v_pages),
                              torch.from_numpy(inp.block_table).cuda(), torch.from_numpy(inp.kv_len).cuda(),
                              D, Hkv, G, dev_status=st2)
    ref, _ = oracle.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                     D, Hkv, G, d, 64)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    err = out.cpu().numpy().astype(np.float64) - ref
    assert np.abs(err).max() <= 2e-2 and np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref)
