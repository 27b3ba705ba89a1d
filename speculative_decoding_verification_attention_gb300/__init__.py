"""Speculative-decoding verification step on one GB300 GPU.

Thin Python binding over the C ABI in ``include/spec_verify.h`` (library
``libspec_verify.so`` built in-tree from ``csrc/``).  The functions below
only marshal arguments -- tensors become device pointers, the current torch
stream becomes the launch stream -- and every step runs in the library's
sm_103a kernels.  PyTorch supplies device memory and streams.

There is no fallback: if the library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "SpecError", "library", "library_path", "verify_attention", "verify_gemm",
    "accept_greedy", "accept_sample", "accept_sample_workspace_size", "attention_workspace_size",
    "gemm_workspace_size", "gemm_plan", "gemm_plan_cluster", "attention_plan", "EXPORTED_SYMBOLS", "DEV_STATUS_BITS",
    "verify_tree_attention", "tree_attention_workspace_size", "accept_tree_greedy", "accept_tree_sample",
    "AdaptiveDraftLength", "accept_sample_logits", "accept_sample_logits_workspace_size",
    "accept_adasd", "accept_adasd_workspace_size", "selftest_bounded_wait",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libspec_verify.so")

EXPORTED_SYMBOLS = (
    "spec_status_string", "spec_version", "spec_verify_attention_workspace_size",
    "spec_verify_attention", "spec_verify_gemm_workspace_size", "spec_verify_gemm",
    "spec_accept_greedy", "spec_accept_sample", "spec_verify_attention_plan",
    "spec_verify_attention_noalloc", "spec_accept_sample_workspace_size", "spec_verify_gemm_plan",
    "spec_verify_gemm_plan_cluster",
    "spec_verify_tree_attention_workspace_size", "spec_verify_tree_attention",
    "spec_accept_tree_greedy", "spec_accept_tree_sample", "spec_adaptive_init", "spec_adaptive_update", "spec_adaptive_draft_len",
    "spec_accept_sample_logits_workspace_size", "spec_accept_sample_logits",
    "spec_accept_adasd_workspace_size", "spec_accept_adasd", "spec_selftest_bounded_wait",
)

DEV_STATUS_BITS = {
    "PAGE_ID": 0x1, "KV_LEN": 0x2, "TIMEOUT": 0x4, "TOKEN_ID": 0x8, "UNIFORM": 0x10,
    "ZERO_MASS": 0x20, "LAUNCH": 0x40, "TREE": 0x80, "LOGITS": 0x100, "PROB": 0x200,
    "INFO_ZERO_RESIDUAL": 0x10000,
}

ATTENTION_KEY_TILE = 128   # SPEC_ATTENTION_KEY_TILE: keys per tile of the KV split

_STATUS = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_UNSUPPORTED",
           3: "SPEC_ERR_WORKSPACE", 4: "SPEC_ERR_CUDA", 5: "SPEC_ERR_TIMEOUT"}


class SpecError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}")


_lock = threading.Lock()
_lib = None


def library():
    """Load libspec_verify.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(
                    f"{library_path} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(library_path)
            P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.spec_status_string.argtypes = [I]
            lib.spec_status_string.restype = ctypes.c_char_p
            lib.spec_version.restype = I
            lib.spec_verify_attention_workspace_size.argtypes = [I, I, I, I, I, I]
            lib.spec_verify_attention_workspace_size.restype = S
            lib.spec_verify_attention.argtypes = [P, P, P, I, P, I, P, I, I, I, I, I, I, F, P, P,
                                                  P, S, P, P]
            lib.spec_verify_attention.restype = I
            lib.spec_verify_gemm_workspace_size.argtypes = [I, I, I]
            lib.spec_verify_gemm_workspace_size.restype = S
            lib.spec_verify_gemm.argtypes = [P, P, P, I, I, I, P, S, P, P]
            lib.spec_verify_gemm.restype = I
            lib.spec_accept_greedy.argtypes = [P, P, I, I, I, P, P, P, P]
            lib.spec_accept_greedy.restype = I
            lib.spec_accept_sample_workspace_size.argtypes = [I, I]
            lib.spec_accept_sample_workspace_size.restype = S
            lib.spec_accept_sample.argtypes = [P, P, P, P, P, I, I, I, P, P, P, S, P, P]
            lib.spec_accept_sample.restype = I
            lib.spec_verify_attention_noalloc.argtypes = [P, P, P, I, P, I, P, I, I, I, I, I, I, F,
                                                          P, P, P, P]
            lib.spec_verify_attention_noalloc.restype = I
            lib.spec_verify_attention_plan.argtypes = [I, P, I, I, I, P, I]
            lib.spec_verify_attention_plan.restype = I
            lib.spec_verify_tree_attention_workspace_size.argtypes = [I, I, I, I, I, I]
            lib.spec_verify_tree_attention_workspace_size.restype = S
            lib.spec_verify_tree_attention.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, F,
                                                       P, P, P, S, P, P]
            lib.spec_verify_tree_attention.restype = I
            lib.spec_accept_tree_greedy.argtypes = [P, P, P, I, I, I, P, P, P, P, P]
            lib.spec_accept_tree_greedy.restype = I
            lib.spec_accept_tree_sample.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P, P, P]
            lib.spec_accept_tree_sample.restype = I
            lib.spec_adaptive_init.argtypes = [P, P, I, F]
            lib.spec_adaptive_init.restype = I
            lib.spec_adaptive_update.argtypes = [P, P, I]
            lib.spec_adaptive_update.restype = I
            lib.spec_adaptive_draft_len.argtypes = [P]
            lib.spec_adaptive_draft_len.restype = I
            lib.spec_verify_gemm_plan.argtypes = [I, I, I, I, P, I]
            lib.spec_verify_gemm_plan.restype = I
            lib.spec_verify_gemm_plan_cluster.argtypes = [I, I, I, I]
            lib.spec_verify_gemm_plan_cluster.restype = I
            lib.spec_accept_sample_logits_workspace_size.argtypes = [I, I, I]
            lib.spec_accept_sample_logits_workspace_size.restype = S
            lib.spec_accept_sample_logits.argtypes = [P, P, P, F, ctypes.c_uint64, I, I, I, P, P, P, S,
                                                      P, P]
            lib.spec_accept_sample_logits.restype = I
            lib.spec_accept_adasd_workspace_size.argtypes = [I, I, I]
            lib.spec_accept_adasd_workspace_size.restype = S
            lib.spec_accept_adasd.argtypes = [P, P, P, P, P, F, F, I, I, I, P, P, P, P, P, P, S, P, P]
            lib.spec_accept_adasd.restype = I
            U64 = ctypes.c_uint64
            lib.spec_selftest_bounded_wait.argtypes = [U64, U64, P, P, P]
            lib.spec_selftest_bounded_wait.restype = I
            _lib = lib
    return _lib


def _check(status, where):
    if status != 0:
        raise SpecError(status, where)


def _dev(t, name, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ attention
def attention_workspace_size(B, D, Hkv, G, head_dim, max_kv_len):
    return int(library().spec_verify_attention_workspace_size(B, D, Hkv, G, head_dim, max_kv_len))


def verify_attention(q, k_pages, v_pages, block_table, kv_len, D, Hkv, G, softmax_scale=None,
                     out=None, lse=None, workspace=None, dev_status=None, stream=None):
    """GQA verify attention over a paged bf16 KV cache.

    q [B, 1+D, Hkv*G, d] bf16; k_pages/v_pages [P, page, Hkv, d] bf16;
    block_table [B, max_pages] int32; kv_len [B] int32 (counts the 1+D
    verify tokens).  Returns out [B, 1+D, Hkv*G, d] fp32 (and fills ``lse``
    [B, 1+D, Hkv*G] fp32 when given).
    """
    import torch
    B, D1, Hq, d = q.shape
    if D1 != D + 1 or Hq != Hkv * G:
        raise ValueError("q shape does not match D/Hkv/G")
    P, page, hk, dk = k_pages.shape
    if hk != Hkv or dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages shape mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, D + 1, Hq, d), dtype=torch.float32, device=q.device)
    max_pages = block_table.shape[1]
    need = attention_workspace_size(B, D, Hkv, G, d, max_pages * page)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = library().spec_verify_attention(
        _dev(q, "q", torch.bfloat16), _dev(k_pages, "k_pages", torch.bfloat16),
        _dev(v_pages, "v_pages", torch.bfloat16), P, _dev(block_table, "block_table", torch.int32),
        max_pages, _dev(kv_len, "kv_len", torch.int32), B, D, Hkv, G, d, page,
        float(softmax_scale), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32, allow_none=True),
        _dev(workspace, "workspace", allow_none=True),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_verify_attention")
    return out


def tree_attention_workspace_size(B, D, Hkv, G, head_dim, max_kv_len):
    return int(library().spec_verify_tree_attention_workspace_size(B, D, Hkv, G, head_dim,
                                                                    max_kv_len))


def verify_tree_attention(q, k_pages, v_pages, block_table, kv_len, tree_parent, D, Hkv, G,
                          softmax_scale=None, out=None, lse=None, workspace=None, dev_status=None,
                          stream=None):
    """Tree verify attention: node k of sequence b attends to the prefix and
    to its root-to-node path.  tree_parent int32 [B, 1+D]; other arguments
    as verify_attention."""
    import torch
    B, D1, Hq, d = q.shape
    if D1 != D + 1 or Hq != Hkv * G:
        raise ValueError("q shape does not match D/Hkv/G")
    P, page, hk, dk = k_pages.shape
    if hk != Hkv or dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages shape mismatch")
    if tuple(tree_parent.shape) != (B, D + 1):
        raise ValueError("tree_parent must be [B, 1+D]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, D + 1, Hq, d), dtype=torch.float32, device=q.device)
    max_pages = block_table.shape[1]
    need = tree_attention_workspace_size(B, D, Hkv, G, d, max_pages * page)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = library().spec_verify_tree_attention(
        _dev(q, "q", torch.bfloat16), _dev(k_pages, "k_pages", torch.bfloat16),
        _dev(v_pages, "v_pages", torch.bfloat16), P, _dev(block_table, "block_table", torch.int32),
        max_pages, _dev(kv_len, "kv_len", torch.int32), _dev(tree_parent, "tree_parent", torch.int32),
        B, D, Hkv, G, d, page, float(softmax_scale), _dev(out, "out", torch.float32),
        _dev(lse, "lse", torch.float32, allow_none=True),
        _dev(workspace, "workspace", allow_none=True),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_verify_tree_attention")
    return out


def attention_plan(kv_len_host, D, Hkv, num_groups, max_segments=None):
    """Segments (group, b, h, tile_begin, tile_end, slot) of the KV split."""
    import numpy as np
    kv = np.ascontiguousarray(kv_len_host, dtype=np.int32)
    if max_segments is None:
        kt = ATTENTION_KEY_TILE
        tiles = int(np.sum((kv.astype(np.int64) + kt - 1) // kt)) * Hkv
        max_segments = tiles + 2 * num_groups + 8
    seg = np.zeros((max_segments, 6), np.int32)
    n = library().spec_verify_attention_plan(len(kv), kv.ctypes.data_as(ctypes.c_void_p), D,
                                             Hkv, num_groups,
                                             seg.ctypes.data_as(ctypes.c_void_p), max_segments)
    if n < 0:
        raise ValueError("spec_verify_attention_plan rejected its arguments")
    return seg[:n]


# ----------------------------------------------------------------------- GEMM
def gemm_workspace_size(M, N, K):
    return int(library().spec_verify_gemm_workspace_size(M, N, K))


def gemm_plan_cluster(M, N, K, num_sms):
    """Cluster size of the planned launch: 2 for CTA pairs (M > 256); for
    M <= 256, 1 for stream-K and S >= 2 for split K over clusters of S."""
    n = library().spec_verify_gemm_plan_cluster(M, N, K, num_sms)
    if n < 0:
        raise ValueError("spec_verify_gemm_plan_cluster rejected its arguments")
    return n


def gemm_plan(M, N, K, num_sms):
    """Segments (cta, tile, kb0, kb1, last, BN) of the planned work split."""
    import numpy as np
    lib = library()
    n = lib.spec_verify_gemm_plan(M, N, K, num_sms, None, 0)
    if n < 0:
        raise ValueError("spec_verify_gemm_plan rejected its arguments")
    seg = np.zeros((max(n, 1), 6), np.int32)
    lib.spec_verify_gemm_plan(M, N, K, num_sms, seg.ctypes.data_as(ctypes.c_void_p), n)
    return seg[:n]


def verify_gemm(x, w, y=None, workspace=None, dev_status=None, stream=None):
    """y[M, N] (bf16) = x[M, K] @ w[N, K]^T with fp32 accumulation.

    ``workspace`` (uint8, ``gemm_workspace_size(M, N, K)`` bytes; 0 for
    M > 256) must be zero-filled before its first use; every call that
    completes leaves it ready for the next (zero it again after a call that
    set a ``dev_status`` bit).  Without one, a zeroed workspace is allocated
    for this call.
    """
    import torch
    M, K = x.shape
    N, K2 = w.shape
    if K2 != K:
        raise ValueError("x/w inner dimensions differ")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = gemm_workspace_size(M, N, K)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    st = library().spec_verify_gemm(
        _dev(x, "x", torch.bfloat16), _dev(w, "w", torch.bfloat16), _dev(y, "y", torch.bfloat16),
        M, N, K, _dev(workspace, "workspace", allow_none=True),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_verify_gemm")
    return y


# ----------------------------------------------------------------- acceptance
def accept_greedy(p, draft, n_accepted=None, token=None, dev_status=None, stream=None):
    """Greedy prefix acceptance; p [B, 1+D, V] fp32, draft [B, D] int32."""
    import torch
    B, D1, V = p.shape
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=p.device)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=p.device)
    st = library().spec_accept_greedy(
        _dev(p, "p", torch.float32), _dev(draft, "draft", torch.int32, allow_none=True), B, D1 - 1,
        V, _dev(n_accepted, "n_accepted", torch.int32), _dev(token, "token", torch.int32),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_accept_greedy")
    return n_accepted, token


def accept_tree_greedy(p, tokens, tree_parent, n_accepted=None, token=None, path=None,
                       dev_status=None, stream=None):
    """Greedy tree acceptance; p [B, 1+D, V] fp32, tokens / tree_parent int32
    [B, 1+D].  Returns (n_accepted, token, path [B, D])."""
    import torch
    B, D1, V = p.shape
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=p.device)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=p.device)
    if path is None:
        path = torch.empty((B, max(D1 - 1, 1)), dtype=torch.int32, device=p.device)
    st = library().spec_accept_tree_greedy(
        _dev(p, "p", torch.float32), _dev(tokens, "tokens", torch.int32),
        _dev(tree_parent, "tree_parent", torch.int32), B, D1 - 1, V,
        _dev(n_accepted, "n_accepted", torch.int32), _dev(token, "token", torch.int32),
        _dev(path, "path", torch.int32), _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_accept_tree_greedy")
    return n_accepted, token, path[:, :D1 - 1]


def accept_tree_sample(p, q, tokens, tree_parent, u_acc, u_res, n_accepted=None, token=None, path=None,
                       dev_status=None, stream=None):
    """Stochastic tree acceptance; p, q [B, 1+D, V] fp32 (q row k: the draft
    distribution of node k's children), tokens / tree_parent int32 [B, 1+D],
    u_acc fp32 [B, 1+D], u_res fp32 [B].  Returns (n_accepted, token,
    path [B, D])."""
    import torch
    B, D1, V = p.shape
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=p.device)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=p.device)
    if path is None:
        path = torch.empty((B, max(D1 - 1, 1)), dtype=torch.int32, device=p.device)
    st = library().spec_accept_tree_sample(
        _dev(p, "p", torch.float32), _dev(q, "q", torch.float32), _dev(tokens, "tokens", torch.int32),
        _dev(tree_parent, "tree_parent", torch.int32), _dev(u_acc, "u_acc", torch.float32),
        _dev(u_res, "u_res", torch.float32), B, D1 - 1, V,
        _dev(n_accepted, "n_accepted", torch.int32), _dev(token, "token", torch.int32),
        _dev(path, "path", torch.int32), _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_accept_tree_sample")
    return n_accepted, token, path[:, :D1 - 1]


def accept_sample_workspace_size(B, V):
    return int(library().spec_accept_sample_workspace_size(B, V))


def accept_sample(p, q, draft, u_acc, u_res, n_accepted=None, token=None, workspace=None,
                  dev_status=None, stream=None):
    """Stochastic acceptance with residual resampling (explicit uniforms).

    ``workspace`` (uint8, ``accept_sample_workspace_size(B, V)`` bytes) is
    scratch; without one it is allocated for this call.
    """
    import torch
    B, D1, V = p.shape
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=p.device)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=p.device)
    need = accept_sample_workspace_size(B, V)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=p.device)
    st = library().spec_accept_sample(
        _dev(p, "p", torch.float32), _dev(q, "q", torch.float32, allow_none=True),
        _dev(draft, "draft", torch.int32, allow_none=True),
        _dev(u_acc, "u_acc", torch.float32, allow_none=True), _dev(u_res, "u_res", torch.float32),
        B, D1 - 1, V, _dev(n_accepted, "n_accepted", torch.int32),
        _dev(token, "token", torch.int32), _dev(workspace, "workspace", allow_none=True),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_accept_sample")
    return n_accepted, token


def accept_sample_logits_workspace_size(B, D, V):
    return int(library().spec_accept_sample_logits_workspace_size(B, D, V))


def accept_sample_logits(target_logits, draft_logits, draft, temperature, seed, n_accepted=None,
                         token=None, workspace=None, dev_status=None, stream=None):
    """Stochastic acceptance from logits: p = softmax(target_logits / T),
    q = softmax(draft_logits / T), uniforms from Philox4x32-10 keyed by
    ``seed`` (spec_accept_sample_logits).

    ``workspace`` (uint8, ``accept_sample_logits_workspace_size(B, D, V)``
    bytes) is scratch; without one it is allocated for this call.
    """
    import torch
    B, D1, V = target_logits.shape
    D = D1 - 1
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    need = accept_sample_logits_workspace_size(B, D, V)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=target_logits.device)
    st = library().spec_accept_sample_logits(
        _dev(target_logits, "target_logits", torch.float32),
        _dev(draft_logits, "draft_logits", torch.float32, allow_none=True),
        _dev(draft, "draft", torch.int32, allow_none=True), float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, B, D, V, _dev(n_accepted, "n_accepted", torch.int32),
        _dev(token, "token", torch.int32), _dev(workspace, "workspace", allow_none=True),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_accept_sample_logits")
    return n_accepted, token


def accept_adasd_workspace_size(B, D, V):
    return int(library().spec_accept_adasd_workspace_size(B, D, V))


def accept_adasd(p, q, draft, u_acc, u_res, tau_entropy, tau_js, n_accepted=None, token=None,
                 draft_len=None, entropy=None, js_distance=None, workspace=None, dev_status=None,
                 stream=None):
    """AdaSD relaxed acceptance (spec_accept_adasd): returns n_accepted,
    token, draft_len (d_eff), entropy [B, D], js_distance [B, D]."""
    import torch
    B, D1, V = p.shape
    D = D1 - 1
    dev = p.device
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=dev)
    if draft_len is None:
        draft_len = torch.empty(B, dtype=torch.int32, device=dev)
    if entropy is None:
        entropy = torch.empty((B, D), dtype=torch.float32, device=dev)
    if js_distance is None:
        js_distance = torch.empty((B, D), dtype=torch.float32, device=dev)
    need = accept_adasd_workspace_size(B, D, V)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    st = library().spec_accept_adasd(
        _dev(p, "p", torch.float32), _dev(q, "q", torch.float32, allow_none=True),
        _dev(draft, "draft", torch.int32, allow_none=True),
        _dev(u_acc, "u_acc", torch.float32, allow_none=True), _dev(u_res, "u_res", torch.float32),
        float(tau_entropy), float(tau_js), B, D, V, _dev(n_accepted, "n_accepted", torch.int32),
        _dev(token, "token", torch.int32), _dev(draft_len, "draft_len", torch.int32),
        _dev(entropy, "entropy", torch.float32) if D else None,
        _dev(js_distance, "js_distance", torch.float32) if D else None,
        _dev(workspace, "workspace", allow_none=True),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(dev_status, "dev_status", allow_none=True), _stream(stream))
    _check(st, "spec_accept_adasd")
    return n_accepted, token, draft_len, entropy, js_distance


# ------------------------------------------------------------ self-test
def selftest_bounded_wait(wait_limit_ns, arrive_after_ns=None, dev_status=None, stream=None):
    """Run the library's bounded mbarrier wait once on the device
    (spec_selftest_bounded_wait): limited to ``wait_limit_ns``, on a barrier
    that is arrived on after ``arrive_after_ns`` (never when None).  Returns
    the device int64 tensor [completed, abort flag, wait duration in ns]."""
    import torch
    res = torch.zeros(3, dtype=torch.int64, device="cuda")
    after = 0xFFFFFFFFFFFFFFFF if arrive_after_ns is None else int(arrive_after_ns)
    st = library().spec_selftest_bounded_wait(int(wait_limit_ns), after, _dev(res, "result"),
                                               _dev(dev_status, "dev_status", allow_none=True),
                                               _stream(stream))
    _check(st, "spec_selftest_bounded_wait")
    return res


# ------------------------------------------------------------ adaptive draft length
class _AdaptiveState(ctypes.Structure):
    _fields_ = [("ema", ctypes.c_float), ("beta", ctypes.c_float), ("rounds", ctypes.c_int),
                ("n_tiers", ctypes.c_int), ("current", ctypes.c_int), ("tiers", ctypes.c_int * 8)]


class AdaptiveDraftLength:
    """Host controller of the draft length (spec_adaptive_*): an EMA of the
    accept length picks one of a few draft-length tiers per round."""

    def __init__(self, tiers=(1, 3, 7), beta=0.9):
        import numpy as np
        self._s = _AdaptiveState()
        t = np.ascontiguousarray(tiers, dtype=np.int32)
        _check(library().spec_adaptive_init(ctypes.byref(self._s), t.ctypes.data_as(ctypes.c_void_p),
                                            len(t), float(beta)), "spec_adaptive_init")

    @property
    def draft_len(self):
        return int(library().spec_adaptive_draft_len(ctypes.byref(self._s)))

    @property
    def ema(self):
        return float(self._s.ema)

    def update(self, n_accepted):
        """n_accepted: host int32 array of the round just verified; returns
        the draft length for the next round."""
        import numpy as np
        a = np.ascontiguousarray(n_accepted, dtype=np.int32)
        d = library().spec_adaptive_update(ctypes.byref(self._s), a.ctypes.data_as(ctypes.c_void_p), a.size)
        if d < 0:
            raise ValueError("spec_adaptive_update rejected its arguments")
        return int(d)
