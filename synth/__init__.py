"""Seeded synthetic inputs for the speculative-decoding verification step.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds input construction only -- random tensors, page tables,
draft tokens drawn from the draft distribution, and the uniforms that the
acceptance rule consumes -- and none of the verification arithmetic itself
(no attention, no GEMM, no accept/reject rule).

Workload recipes follow the five verification-step configurations:

* tiny step: B=1, one KV head, G=4, head_dim=64, contiguous KV of 256
  tokens, D=3; acceptance on V=1000 with target logits N(0, 2^2) and draft
  logits = target + N(0, 0.5^2).
* throughput-regime attention: B=16, Hkv=8, G=8, head_dim=128, L=32768, D=15.
* large-group attention: B=8, Hkv=4, G=32, head_dim=128, L=131072,
  D in {0,1,3,4,7,15}.
* batched acceptance: B=256, D=7, V=131072, target logits N(0, 3^2),
  draft logits = target + N(0, sigma^2) with sigma tuned to an acceptance
  rate alpha.
* full step: B=64, L_b ~ U{4096..131072}, 64-token pages in a random
  permutation, Hkv=8, G=8, head_dim=128, D=7; verify GEMM M=B(1+D) in
  {8..4096} x N=K=6144 with W ~ N(0, 0.02^2), x ~ N(0, 1).

Random numbers the acceptance rule draws are produced here by a
counter-based Philox4x32-10 generator (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11) and passed to both
sides as explicit fp32 arrays.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "philox4x32_10", "philox_uniform", "acceptance_uniforms",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "AttentionInputs",
    "attention_inputs", "paged_layout", "accept_inputs", "gemm_inputs",
    "draw_from_rows", "tune_sigma_for_alpha", "tree_sample_inputs", "STREAM_ACCEPT",
    "STREAM_RESAMPLE", "STREAM_DRAFT",
]

# ---------------------------------------------------------------------------
# Philox4x32-10 (SC'11, section 3: the Philox S-box uses two 32x32->64
# multiplications per round, a Weyl-sequence key schedule, and 10 rounds for
# the "-10" variant).  Constants are the published multipliers and the key
# increments (golden ratio and sqrt(3)-1 in 32-bit fixed point).
# ---------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = 0x9E3779B9
_PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

STREAM_ACCEPT = 0     # u_acc[b, i]: counter (b, i, 0, 0)
STREAM_RESAMPLE = 1   # u_res[b]:    counter (b, 0, 1, 0)
STREAM_DRAFT = 2      # draft draw:  counter (b, i, 2, 0)


def philox4x32_10(c0, c1, c2, c3, key):
    """Philox4x32 with 10 rounds on uint32 counter words (broadcastable).

    ``key`` is a 64-bit integer split into (k0 = low word, k1 = high word).
    Returns four uint32 arrays.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK32 for c in (c0, c1, c2, c3))
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    c0, c1, c2, c3 = (c.copy() for c in (c0, c1, c2, c3))
    k0 = int(key) & 0xFFFFFFFF
    k1 = (int(key) >> 32) & 0xFFFFFFFF
    for _ in range(10):
        p0 = c0 * _PHILOX_M0
        p1 = c2 * _PHILOX_M1
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + _PHILOX_W0) & 0xFFFFFFFF
        k1 = (k1 + _PHILOX_W1) & 0xFFFFFFFF
    return tuple(c.astype(np.uint32) for c in (c0, c1, c2, c3))


def philox_uniform(seed, c0, c1, stream):
    """fp32 uniform in [0, 1): the top 24 bits of Philox word 0, times 2^-24.

    Every value is exactly representable in fp32 and fp64.
    """
    x0, _, _, _ = philox4x32_10(c0, c1, stream, 0, seed)
    return ((x0 >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


def acceptance_uniforms(seed, B, D, b_offset=0):
    """(u_acc [B, D], u_res [B]) as fp32 for sequences b_offset..b_offset+B-1."""
    b = np.arange(b_offset, b_offset + B, dtype=np.uint64)
    i = np.arange(max(D, 1), dtype=np.uint64)
    u_acc = philox_uniform(seed, b[:, None], i[None, :], STREAM_ACCEPT)[:, :D]
    u_res = philox_uniform(seed, b, np.zeros_like(b), STREAM_RESAMPLE)
    return np.ascontiguousarray(u_acc, dtype=np.float32), u_res.astype(np.float32)


# ---------------------------------------------------------------------------
# bf16 bit patterns (round to nearest even), stored as uint16.
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    out = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# Attention inputs: Q [B, 1+D, Hq, d], paged K/V [P, page, Hkv, d] as bf16
# bits, block_table [B, max_pages] int32, kv_len [B] int32.  Row (i, g) of KV
# head h reads query head h*G + g.
# ---------------------------------------------------------------------------
class AttentionInputs(dict):
    __getattr__ = dict.__getitem__


def paged_layout(kv_len, page_size, rng, permute=True, spare_pages=0):
    """Page table for sequences of lengths ``kv_len``.

    Returns (block_table [B, max_pages] int32, num_pages).  Entries past a
    sequence's last page are filled with -1 so that any read of them is
    caught by the kernel's page-id check.
    """
    kv_len = np.asarray(kv_len, dtype=np.int64)
    n_pages = (kv_len + page_size - 1) // page_size
    total = int(n_pages.sum()) + int(spare_pages)
    ids = rng.permutation(total) if permute else np.arange(total)
    max_pages = int(max(1, n_pages.max()))
    table = np.full((len(kv_len), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(n_pages):
        table[b, :n] = ids[off:off + n]
        off += n
    return table, total


def attention_inputs(seed, B, Hkv, G, head_dim, D, kv_len, page_size=64,
                     permute=True, q_std=1.0, kv_std=1.0):
    """Host (numpy) attention inputs for small cases; values ~ N(0, std^2)."""
    rng = np.random.default_rng(seed)
    kv_len = np.broadcast_to(np.asarray(kv_len, dtype=np.int32), (B,)).copy()
    Hq = Hkv * G
    table, P = paged_layout(kv_len, page_size, rng, permute)
    q = f32_to_bf16_bits(rng.standard_normal((B, 1 + D, Hq, head_dim), dtype=np.float32) * q_std)
    k = f32_to_bf16_bits(rng.standard_normal((P, page_size, Hkv, head_dim), dtype=np.float32) * kv_std)
    v = f32_to_bf16_bits(rng.standard_normal((P, page_size, Hkv, head_dim), dtype=np.float32) * kv_std)
    return AttentionInputs(q=q, k_pages=k, v_pages=v, block_table=table, kv_len=kv_len,
                           B=B, D=D, Hkv=Hkv, G=G, head_dim=head_dim, page_size=page_size,
                           num_pages=P)


# ---------------------------------------------------------------------------
# Acceptance inputs.
# ---------------------------------------------------------------------------
def _softmax64(logits):
    z = logits - logits.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def draw_from_rows(probs, u):
    """Inverse-CDF draw of one index per row of ``probs`` (fp64 cumulative).

    This is the drafter's own sampling, used to synthesise draft tokens.
    """
    c = np.cumsum(np.asarray(probs, dtype=np.float64), axis=-1)
    t = np.asarray(u, dtype=np.float64)[..., None] * c[..., -1:]
    idx = (c <= t).sum(axis=-1)
    return np.minimum(idx, probs.shape[-1] - 1).astype(np.int32)


def tune_sigma_for_alpha(alpha, V, seed=1234, rows=64, target_std=3.0, tol=0.005):
    """Bisection on the draft-logit noise sigma so that the mean over rows of
    sum_v min(p, q) equals ``alpha`` within ``tol`` on a fixed seed."""
    rng = np.random.default_rng(seed)
    t = rng.standard_normal((rows, V)) * target_std
    noise = rng.standard_normal((rows, V))
    p = _softmax64(t)

    def overlap(sig):
        q = _softmax64(t + sig * noise)
        return float(np.minimum(p, q).sum(axis=-1).mean())

    lo, hi = 0.0, 20.0
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if overlap(mid) > alpha:
            lo = mid
        else:
            hi = mid
        if abs(overlap(mid) - alpha) < tol * 0.2:
            break
    sig = 0.5 * (lo + hi)
    return sig, overlap(sig)


def accept_inputs(seed, B, D, V, target_std=2.0, draft_noise=0.5, mode="sample",
                  b_offset=0, chunk=32):
    """p [B, 1+D, V], q [B, D, V] (fp32 softmax of fp64 logits), drafts
    [B, D] int32, u_acc [B, D], u_res [B] fp32.

    Target logits ~ N(0, target_std^2); draft logits = target logits (first D
    positions) + N(0, draft_noise^2).  mode="sample": draft i is drawn from
    q[b, i] with Philox stream 2; mode="greedy": draft i = argmax q[b, i]
    (lowest index on ties); mode="both" returns both as draft_sample /
    draft_greedy (and draft = draft_sample).  Generated in chunks of
    sequences to bound host memory.
    """
    rng = np.random.default_rng(seed)
    p = np.empty((B, 1 + D, V), np.float32)
    q = np.empty((B, D, V), np.float32)
    for s0 in range(0, B, chunk):
        s1 = min(B, s0 + chunk)
        t = rng.standard_normal((s1 - s0, 1 + D, V)) * target_std
        p[s0:s1] = _softmax64(t)
        if D:
            q[s0:s1] = _softmax64(t[:, :D, :] + rng.standard_normal((s1 - s0, D, V)) * draft_noise)
        del t
    out = dict(p=p, q=q, B=B, D=D, V=V)
    b = np.arange(b_offset, b_offset + B, dtype=np.uint64)
    i = np.arange(max(D, 1), dtype=np.uint64)
    if mode in ("sample", "both"):
        ud = philox_uniform(seed, b[:, None], i[None, :], STREAM_DRAFT)[:, :D]
        ds = np.empty((B, D), np.int32)
        for s0 in range(0, B, chunk):
            ds[s0:s0 + chunk] = draw_from_rows(q[s0:s0 + chunk], ud[s0:s0 + chunk])
        out["draft_sample"] = ds
    if mode in ("greedy", "both"):
        out["draft_greedy"] = np.argmax(q, axis=-1).astype(np.int32) if D else np.zeros((B, 0), np.int32)
    if mode not in ("sample", "greedy", "both"):
        raise ValueError(mode)
    out["draft"] = out["draft_greedy"] if mode == "greedy" else out["draft_sample"]
    out["u_acc"], out["u_res"] = acceptance_uniforms(seed, B, D, b_offset)
    return out


def logits_inputs(seed, B, D, V, target_std=3.0, draft_noise=0.5, temperature=1.0, masked=0,
                  b_offset=0, chunk=16):
    """Target logits zp [B, 1+D, V] and draft logits zq [B, D, V] (fp32),
    drafts [B, D] int32.

    zp ~ N(0, target_std^2); zq = zp (first D positions) + N(0, draft_noise^2).
    ``masked`` vocabulary entries per sequence (the same positions in every
    row of it) are -inf in both.  Draft i is drawn from the fp64 softmax of
    zq[b, i] / temperature with Philox stream 2 (the drafter's own sampling).
    Generated in chunks of sequences to bound host memory.
    """
    rng = np.random.default_rng(seed)
    zp = np.empty((B, 1 + D, V), np.float32)
    zq = np.empty((B, D, V), np.float32)
    draft = np.empty((B, D), np.int32)
    b = np.arange(b_offset, b_offset + B, dtype=np.uint64)
    i = np.arange(max(D, 1), dtype=np.uint64)
    ud = philox_uniform(seed, b[:, None], i[None, :], STREAM_DRAFT)[:, :D]
    for s0 in range(0, B, chunk):
        s1 = min(B, s0 + chunk)
        t = (rng.standard_normal((s1 - s0, 1 + D, V), dtype=np.float32) * np.float32(target_std))
        zp[s0:s1] = t
        if D:
            zq[s0:s1] = t[:, :D, :] + rng.standard_normal((s1 - s0, D, V), dtype=np.float32) * np.float32(
                draft_noise)
        if masked:
            for s in range(s0, s1):
                cols = rng.choice(V, size=min(masked, V - 1), replace=False)
                zp[s][:, cols] = -np.inf
                zq[s][:, cols] = -np.inf
        if D:
            probs = _softmax64(zq[s0:s1].astype(np.float64) / temperature)
            draft[s0:s1] = draw_from_rows(probs, ud[s0:s1])
            del probs
        del t
    return dict(zp=zp, zq=zq, draft=draft, B=B, D=D, V=V, temperature=temperature, seed=seed)


def gemm_inputs(seed, M, N, K, w_std=0.02):
    rng = np.random.default_rng(seed)
    x = f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * w_std)
    return x, w


def full_step_kv_lengths(seed, B=64, lo=4096, hi=131072):
    """Seeded integer KV lengths L_b ~ U{lo..hi} for the full-step workload."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=B).astype(np.int32)


# ---------------------------------------------------------------------------
# Device-side generation for the large workloads (torch is used for memory
# and its own seeded normal generator only).
# ---------------------------------------------------------------------------
def attention_inputs_device(seed, B, Hkv, G, head_dim, D, kv_len, page_size=64,
                            permute=True, device="cuda"):
    import torch

    rng = np.random.default_rng(seed)
    kv_len = np.broadcast_to(np.asarray(kv_len, dtype=np.int32), (B,)).copy()
    table, P = paged_layout(kv_len, page_size, rng, permute)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    Hq = Hkv * G

    def randn_bf16(shape):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        step = 1 << 28
        for s in range(0, flat.numel(), step):
            n = min(step, flat.numel() - s)
            flat[s:s + n] = torch.randn(n, generator=gen, device=device,
                                        dtype=torch.float32).to(torch.bfloat16)
        return out

    q = randn_bf16((B, 1 + D, Hq, head_dim))
    k = randn_bf16((P, page_size, Hkv, head_dim))
    v = randn_bf16((P, page_size, Hkv, head_dim))
    return AttentionInputs(q=q, k_pages=k, v_pages=v,
                           block_table=torch.from_numpy(table).to(device),
                           kv_len=torch.from_numpy(kv_len).to(device),
                           block_table_host=table, kv_len_host=kv_len,
                           B=B, D=D, Hkv=Hkv, G=G, head_dim=head_dim,
                           page_size=page_size, num_pages=P)


def bits_from_device(t):
    """Copy a device bf16 tensor back as uint16 bit patterns (numpy)."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def softmax_rows_fp32(logits):
    """fp32 probabilities from fp64 logits (input synthesis helper)."""
    return _softmax64(np.asarray(logits, dtype=np.float64)).astype(np.float32)


def log2_ceil(x):
    return int(math.ceil(math.log2(max(1, x))))


# ---------------------------------------------------------------------------
# Draft trees.
# ---------------------------------------------------------------------------
def tree_sample_inputs(seed, B, D, V, kind="random", target_std=2.0, draft_noise=0.5):
    """Inputs of the stochastic tree acceptance: p, q float32 [B, 1+D, V]
    (fp32 softmax of fp64 logits; target logits ~ N(0, target_std^2) per
    node, draft logits = target + N(0, draft_noise^2)), parent int32
    [B, 1+D] (``tree_parents``), tokens int32 [B, 1+D] where node k's token
    is drawn from q[b, parent[k]] with Philox stream 2, counter (b, k)
    (siblings are independent draws; entry 0 is 0), u_acc float32 [B, 1+D]
    from counter (b, k, 0, 0) and u_res float32 [B] from (b, 0, 1, 0)."""
    rng = np.random.default_rng(seed)
    T = 1 + D
    t = rng.standard_normal((B, T, V)) * target_std
    p = _softmax64(t).astype(np.float32)
    q = _softmax64(t + rng.standard_normal((B, T, V)) * draft_noise).astype(np.float32)
    parent = tree_parents(seed + 1, B, T, kind)
    b = np.arange(B, dtype=np.uint64)
    k = np.arange(T, dtype=np.uint64)
    ud = philox_uniform(seed, b[:, None], k[None, :], STREAM_DRAFT)
    tokens = np.zeros((B, T), np.int32)
    for kk in range(1, T):
        rows = q[np.arange(B), parent[:, kk]]
        tokens[:, kk] = draw_from_rows(rows, ud[:, kk])
    u_acc = philox_uniform(seed, b[:, None], k[None, :], STREAM_ACCEPT).astype(np.float32)
    u_res = philox_uniform(seed, b, np.zeros_like(b), STREAM_RESAMPLE).astype(np.float32)
    return dict(p=p, q=q, parent=parent, tokens=tokens, u_acc=u_acc, u_res=u_res)


def tree_parents(seed, B, T, kind="random"):
    """Parent arrays int32 [B, T] of draft trees in topological order
    (parent[:, 0] = -1, 0 <= parent[b, k] < k).

    kind: "chain" (k - 1), "star" (every node a child of the root),
    "random" (uniform earlier node, a fresh tree per sequence), or "wide"
    (a fixed tree shaped like the static trees of multi-head drafters:
    several candidates at the first level, fewer below).
    """
    par = np.empty((B, T), np.int32)
    par[:, 0] = -1
    if kind == "chain":
        par[:, 1:] = np.arange(T - 1)
    elif kind == "star":
        par[:, 1:] = 0
    elif kind == "random":
        rng = np.random.default_rng(seed)
        for k in range(1, T):
            par[:, k] = rng.integers(0, k, size=B)
    elif kind == "wide":
        # level sizes 4, 3, 2, 1, ... : node k's parent is the first node of
        # the previous level that still has room (at most 3 children each)
        shape = [0]
        levels = [[0]]
        k = 1
        width = 4
        while k < T:
            prev = levels[-1]
            cur = []
            for c in range(width):
                if k >= T:
                    break
                shape.append(prev[min(c // 3, len(prev) - 1)] if c >= 1 else prev[0])
                cur.append(k)
                k += 1
            levels.append(cur)
            width = max(1, width - 1)
        par[:, :] = np.asarray(shape[:T], np.int32)[None, :]
        par[:, 0] = -1
    else:
        raise ValueError(kind)
    return par


def tree_depths(parent):
    """Depth of every node (root 0) of int32 parent arrays [B, T]."""
    B, T = parent.shape
    dep = np.zeros((B, T), np.int32)
    for k in range(1, T):
        dep[:, k] = dep[np.arange(B), parent[:, k]] + 1
    return dep
