"""Pins for the oracle's verify attention (CPU only).

The oracle is checked against things other than itself:
  * torch's fp64 scaled-dot-product attention with an explicitly
    materialised boolean mask (a library routine on a contiguous copy of the
    cache gathered here through the page table);
  * D = 0 equals ordinary decode attention over all kv_len keys;
  * row i of a verify call equals a D = 0 call over the prefix L - D + i
    (the drafts reuse the KV cache: "Draft length and attention
    performance", co-design blog);
  * paged equals contiguous under a random page permutation;
  * closed forms: a one-hot score returns that key's value row, constant keys
    return the mean of the visible value rows.
"""
import numpy as np
import pytest
import torch

import synth


def gather_contiguous(inp, b, h):
    """Keys/values of sequence b, head h as fp64 [L, d] (numpy gather)."""
    L = int(inp.kv_len[b])
    ps = inp.page_size
    j = np.arange(L)
    pages = inp.block_table[b, j // ps]
    k = synth.bf16_bits_to_f32(inp.k_pages[pages, j % ps, h, :]).astype(np.float64)
    v = synth.bf16_bits_to_f32(inp.v_pages[pages, j % ps, h, :]).astype(np.float64)
    return k, v


def torch_reference(inp, scale):
    """fp64 SDPA with a materialised bottom-right causal mask."""
    B, D, Hkv, G, d = inp.B, inp.D, inp.Hkv, inp.G, inp.head_dim
    q = synth.bf16_bits_to_f32(inp.q).astype(np.float64)
    out = np.empty(q.shape)
    for b in range(B):
        L = int(inp.kv_len[b])
        for h in range(Hkv):
            k, v = gather_contiguous(inp, b, h)
            # queries of this KV head: [(1+D)*G, d], row (i, g)
            qq = q[b, :, h * G:(h + 1) * G, :].reshape((1 + D) * G, d)
            i_of_row = np.repeat(np.arange(1 + D), G)
            mask = np.arange(L)[None, :] < (L - D + i_of_row)[:, None]
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(qq)[None, None], torch.from_numpy(k)[None, None],
                torch.from_numpy(v)[None, None], attn_mask=torch.from_numpy(mask)[None, None],
                scale=scale)
            out[b, :, h * G:(h + 1) * G, :] = o[0, 0].numpy().reshape(1 + D, G, d)
    return out


CASES = [
    # B, Hkv, G, d, D, kv_len, page
    (1, 1, 4, 64, 3, [64], 16),
    (2, 2, 3, 32, 2, [37, 50], 16),
    (2, 3, 2, 16, 0, [5, 33], 8),
    (1, 2, 4, 16, 5, [6], 4),      # kv_len == 1 + D: row 0 sees one key
    (3, 1, 1, 8, 1, [2, 17, 40], 32),
]


@pytest.mark.parametrize("B,Hkv,G,d,D,kv_len,page", CASES)
def test_matches_library_sdpa(oracle_lib, B, Hkv, G, d, D, kv_len, page):
    inp = synth.attention_inputs(11, B, Hkv, G, d, D, kv_len, page_size=page)
    scale = 1.0 / np.sqrt(d)
    out, lse = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                           inp.kv_len, D, Hkv, G, d, page, scale)
    ref = torch_reference(inp, scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_lse_is_log_partition(oracle_lib):
    from scipy.special import logsumexp
    inp = synth.attention_inputs(5, 2, 2, 2, 16, 2, [20, 9], page_size=4)
    scale = 0.3
    _, lse = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                         inp.kv_len, 2, 2, 2, 16, 4, scale)
    q = synth.bf16_bits_to_f32(inp.q).astype(np.float64)
    for b in range(2):
        L = int(inp.kv_len[b])
        for h in range(2):
            k, _ = gather_contiguous(inp, b, h)
            for i in range(3):
                for g in range(2):
                    s = scale * (k[:L - 2 + i] @ q[b, i, h * 2 + g])
                    assert abs(lse[b, i, h * 2 + g] - logsumexp(s)) < 1e-12


def test_d0_is_decode_attention(oracle_lib):
    """D = 0 reduces to plain decode attention over every key."""
    inp = synth.attention_inputs(3, 2, 2, 4, 32, 0, [45, 64], page_size=16)
    out, _ = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                         inp.kv_len, 0, 2, 4, 32, 16)
    q = synth.bf16_bits_to_f32(inp.q).astype(np.float64)
    for b in range(2):
        for h in range(2):
            k, v = gather_contiguous(inp, b, h)
            for g in range(4):
                o = torch.nn.functional.scaled_dot_product_attention(
                    torch.from_numpy(q[b, 0, h * 4 + g])[None, None, None],
                    torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None])
                np.testing.assert_allclose(out[b, 0, h * 4 + g], o[0, 0, 0].numpy(),
                                           rtol=1e-12, atol=1e-13)


def test_row_i_equals_prefix_decode(oracle_lib):
    """Row i of a D-draft verify equals D=0 attention over prefix L-D+i."""
    B, Hkv, G, d, D = 2, 2, 4, 32, 5
    inp = synth.attention_inputs(7, B, Hkv, G, d, D, [70, 41], page_size=16)
    out, lse = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                           inp.kv_len, D, Hkv, G, d, 16)
    for b in range(B):
        L = int(inp.kv_len[b])
        for i in range(1 + D):
            q1 = np.ascontiguousarray(inp.q[b:b + 1, i:i + 1])
            o1, l1 = oracle_lib.verify_attention(q1, inp.k_pages, inp.v_pages,
                                                 inp.block_table[b:b + 1],
                                                 np.array([L - D + i], np.int32), 0, Hkv, G,
                                                 d, 16)
            assert np.array_equal(o1[0, 0], out[b, i])   # bit-exact in fp64
            assert np.array_equal(l1[0, 0], lse[b, i])


def test_paged_equals_contiguous(oracle_lib):
    B, Hkv, G, d, D = 3, 2, 2, 16, 3
    lens = [33, 64, 18]
    paged = synth.attention_inputs(9, B, Hkv, G, d, D, lens, page_size=8, permute=True)
    o_p, l_p = oracle_lib.verify_attention(paged.q, paged.k_pages, paged.v_pages,
                                           paged.block_table, paged.kv_len, D, Hkv, G, d, 8)
    # re-pack each sequence contiguously into one big page
    Lmax = max(lens)
    k = np.zeros((B, Lmax, Hkv, d), np.uint16)
    v = np.zeros((B, Lmax, Hkv, d), np.uint16)
    for b in range(B):
        j = np.arange(lens[b])
        pages = paged.block_table[b, j // 8]
        k[b, :lens[b]] = paged.k_pages[pages, j % 8]
        v[b, :lens[b]] = paged.v_pages[pages, j % 8]
    table = np.arange(B, dtype=np.int32)[:, None]
    o_c, l_c = oracle_lib.verify_attention(paged.q, k, v, table, paged.kv_len, D, Hkv, G, d,
                                           Lmax)
    assert np.array_equal(o_p, o_c) and np.array_equal(l_p, l_c)


def test_one_hot_score_returns_value_row(oracle_lib):
    d, L, D = 16, 24, 2
    inp = synth.attention_inputs(1, 1, 1, 1, d, D, [L], page_size=8, permute=False)
    q = np.zeros((1, 1 + D, 1, d), np.float32)
    q[..., 0] = 64.0
    k = np.zeros((inp.num_pages, 8, 1, d), np.float32)
    hot = 5
    k[hot // 8, hot % 8, 0, 0] = 64.0     # score 4096/4 = 1024 vs 0 elsewhere
    out, _ = oracle_lib.verify_attention(synth.f32_to_bf16_bits(q), synth.f32_to_bf16_bits(k),
                                         inp.v_pages, inp.block_table, inp.kv_len, D, 1, 1, d,
                                         8)
    vrow = synth.bf16_bits_to_f32(inp.v_pages[hot // 8, hot % 8, 0]).astype(np.float64)
    for i in range(1 + D):
        np.testing.assert_allclose(out[0, i, 0], vrow, rtol=0, atol=1e-300)


def test_constant_keys_give_mean_of_visible_values(oracle_lib):
    d, L, D = 8, 30, 4
    inp = synth.attention_inputs(2, 1, 1, 2, d, D, [L], page_size=8, permute=True)
    k = np.full_like(inp.k_pages, synth.f32_to_bf16_bits(np.float32(0.75)))
    out, _ = oracle_lib.verify_attention(inp.q, k, inp.v_pages, inp.block_table, inp.kv_len, D,
                                         1, 2, d, 8)
    _, v = gather_contiguous(inp, 0, 0)
    for i in range(1 + D):
        mean = v[:L - D + i].mean(axis=0)
        for g in range(2):
            np.testing.assert_allclose(out[0, i, g], mean, rtol=1e-13, atol=1e-14)


def test_rows_api_matches_full(oracle_lib):
    inp = synth.attention_inputs(4, 2, 2, 2, 16, 3, [40, 25], page_size=8)
    full, lse = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                            inp.kv_len, 3, 2, 2, 16, 8)
    rows = np.array([[1, 3, 1, 0], [0, 0, 0, 1], [1, 2, 0, 1]], np.int32)
    sub, sl = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                          inp.kv_len, 3, 2, 2, 16, 8, rows=rows)
    for n, (b, i, h, g) in enumerate(rows):
        assert np.array_equal(sub[n], full[b, i, h * 2 + g])
        assert sl[n] == lse[b, i, h * 2 + g]


def test_bad_page_id_is_reported(oracle_lib):
    inp = synth.attention_inputs(4, 1, 1, 1, 8, 1, [16], page_size=8)
    table = inp.block_table.copy()
    table[0, 1] = inp.num_pages + 3
    with pytest.raises(ValueError):
        oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, table, inp.kv_len, 1, 1,
                                    1, 8, 8)
