"""The allocation-free attention entry point (GPU).

spec_verify_attention_noalloc serves callers that cannot give the library a
device buffer (an engine plugin whose host framework owns every byte of
device memory, or a serving loop that must not call cudaMalloc because it
would synchronise the device).  It takes its scratch from a fixed array
inside the library.  This test calls it through the C ABI twice in a row,
on different problems so the second call reuses scratch the first left
behind, and checks each result against spec_verify_attention with a
caller-provided workspace, within the attention tolerance.  It lives in a
file collected last and builds what it needs, so it also passes alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 1e-3


@pytest.fixture(scope="module")
def sv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


def dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def call_noalloc(lib, t, D, Hkv, G, d, page, num_pages, stream):
    import torch
    B = t["kv"].shape[0]
    out = torch.full((B, D + 1, Hkv * G, d), float("nan"), device="cuda")
    lse = torch.full((B, D + 1, Hkv * G), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    st = lib.spec_verify_attention_noalloc(
        P(t["q"].data_ptr()), P(t["k"].data_ptr()), P(t["v"].data_ptr()), num_pages,
        P(t["bt"].data_ptr()), t["bt"].shape[1], P(t["kv"].data_ptr()), B, D, Hkv, G, d, page,
        1.0 / np.sqrt(d), P(out.data_ptr()), P(lse.data_ptr()), P(status.data_ptr()),
        P(stream.cuda_stream))
    return st, out, lse, status


@pytest.mark.parametrize("first,second", [
    ((3, 2, 8, 128, 7, [900, 3000, 77], 64), (2, 4, 32, 128, 4, [5000, 1200], 64)),
])
def test_noalloc_matches_workspace_entry_point(sv, first, second):
    import torch
    lib = sv.library()
    stream = torch.cuda.current_stream()
    for seed, (B, Hkv, G, d, D, lens, page) in enumerate((first, second)):
        inp = synth.attention_inputs(300 + seed, B, Hkv, G, d, D, lens, page_size=page)
        t = dict(q=dev_bf16(inp.q), k=dev_bf16(inp.k_pages), v=dev_bf16(inp.v_pages),
                 bt=torch.from_numpy(inp.block_table).cuda(), kv=torch.from_numpy(inp.kv_len).cuda())
        st, out, lse, status = call_noalloc(lib, t, D, Hkv, G, d, page, inp.num_pages, stream)
        assert st == 0
        ref_lse = torch.empty_like(lse)
        ref = sv.verify_attention(t["q"], t["k"], t["v"], t["bt"], t["kv"], D, Hkv, G, lse=ref_lse)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o, r = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(o).all()
        assert np.abs(o - r).max() <= MAX_ABS
        assert np.linalg.norm(o - r) / np.linalg.norm(r) <= REL_L2
        lo, lr = lse.double().cpu().numpy(), ref_lse.double().cpu().numpy()
        assert np.abs(lo - lr).max() <= MAX_ABS


def test_noalloc_scratch_covers_supported_shapes_and_rejects_bad_ones(sv):
    lib = sv.library()
    limit = 24 << 20   # SPEC_NOALLOC_SCRATCH_BYTES
    # the largest supported problems fit in the fixed scratch on this device
    for head_dim, G, D in ((128, 16, 63), (128, 1024, 0), (64, 128, 7), (128, 8, 7)):
        assert 0 < sv.attention_workspace_size(64, D, 8, G, head_dim, 131072) <= limit
    # an unsupported head_dim is rejected before anything is launched
    P = ctypes.c_void_p
    fake = P(0x7F0000001000)
    assert lib.spec_verify_attention_noalloc(fake, fake, fake, 1, fake, 1, fake, 1, 0, 1, 1, 96,
                                             16, 0.1, fake, None, None, None) == 2
