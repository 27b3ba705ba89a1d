"""CUDA-graph tiers of the verification step (GPU).

One graph per draft length D in {1, 3, 7}; replaying a tier's graph must
give exactly what launching the same step eagerly gives, and a controller
driven loop can switch tiers between rounds.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


class Tier:
    """Static buffers of one tier's step: verify attention, one linear
    layer at GEMM-M = B(1+D), stochastic acceptance."""

    def __init__(self, sv, D, B=4, Hkv=2, G=4, L=2048, V=4096, N=512, seed=0):
        import torch
        self.sv, self.D, self.B, self.Hkv, self.G = sv, D, B, Hkv, G
        self.attn = synth.attention_inputs_device(seed + D, B, Hkv, G, 128, D, L, page_size=64)
        self.out = torch.empty((B, D + 1, Hkv * G, 128), device="cuda")
        self.ws_a = torch.empty(sv.attention_workspace_size(B, D, Hkv, G, 128, L), dtype=torch.uint8,
                                device="cuda")
        x, w = synth.gemm_inputs(seed + 10 + D, B * (D + 1), N, 512)
        to = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        self.x, self.w = to(x), to(w)
        self.y = torch.empty((B * (D + 1), N), dtype=torch.bfloat16, device="cuda")
        self.ws_g = torch.zeros(max(256, sv.gemm_workspace_size(B * (D + 1), N, 512)), dtype=torch.uint8,
                                device="cuda")
        acc = synth.accept_inputs(seed + 20 + D, B, D, V, mode="sample")
        self.acc = {k: torch.from_numpy(np.ascontiguousarray(acc[k])).cuda()
                    for k in ("p", "q", "draft", "u_acc", "u_res")}
        self.na = torch.empty(B, dtype=torch.int32, device="cuda")
        self.tk = torch.empty(B, dtype=torch.int32, device="cuda")
        self.ws_s = torch.empty(sv.accept_sample_workspace_size(B, V), dtype=torch.uint8, device="cuda")

    def step(self):
        a, c = self.attn, self.acc
        self.sv.verify_attention(a.q, a.k_pages, a.v_pages, a.block_table, a.kv_len, self.D, self.Hkv, self.G,
                                 out=self.out, workspace=self.ws_a)
        self.sv.verify_gemm(self.x, self.w, y=self.y, workspace=self.ws_g)
        self.sv.accept_sample(c["p"], c["q"], c["draft"], c["u_acc"], c["u_res"], self.na, self.tk,
                              workspace=self.ws_s)

    def results(self):
        return [t.clone() for t in (self.out, self.y, self.na, self.tk)]


def test_graph_tiers_replay_exactly(sv):
    import torch
    from speculative_decoding_verification_attention_gb300.graphs import TierGraphs
    tiers = {D: Tier(sv, D) for D in (1, 3, 7)}
    eager = {}
    for D, t in tiers.items():
        t.step()
        torch.cuda.synchronize()
        eager[D] = t.results()
    graphs = TierGraphs(lambda D: tiers[D].step(), tiers=(1, 3, 7))
    ctl = sv.AdaptiveDraftLength((1, 3, 7), beta=0.5)
    seen = set()
    for r in range(9):
        D = ctl.draft_len
        seen.add(D)
        for x in tiers[D].results():
            x.zero_()
        graphs.replay(D)
        torch.cuda.synchronize()
        for got, ref in zip(tiers[D].results(), eager[D]):
            assert torch.equal(got, ref)
        # drive the controller with a synthetic acceptance pattern
        n = np.full(4, [0, D, 1, D // 2, 0, 0, D, D, 0][r], np.int32)
        ctl.update(n)
    assert len(seen) >= 2
