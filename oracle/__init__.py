"""fp64 CPU parity oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  The
product library never imports this package, and this package imports
nothing from the product.

The arithmetic lives in ``spec_oracle.c`` (plain C, fp64, optional OpenMP
over independent units); this module compiles it with gcc on first use and
wraps it for numpy arrays.  Every function cites the page passage it
follows in the C source.

Parity status of each function (what pins it, in tests/test_oracle_*.py):
  verify_attention  brute force vs torch's fp64 scaled-dot-product attention
                    with a materialised mask; D=0 equals decode attention;
                    row i equals D=0 over the prefix L-D+i; paged equals
                    contiguous; one-hot and constant-key closed forms.
  gemm              numpy fp64 matmul (library routine).
  accept_greedy     brute force over all drafts of a toy target model:
                    emitted tokens equal plain greedy decoding.
  accept_sample     exact enumeration on a toy model (emitted sequence law
                    equals the target's), tau closed form, chi-square.
  tree_attention    a chain tree equals verify_attention bit for bit; every
                    node's row equals decode attention over the prefix
                    followed by its root-to-node path (gathered cache);
                    brute force vs torch's fp64 attention with a
                    materialised tree mask.
  accept_tree_greedy  a chain tree equals accept_greedy; brute force over
                    the accepted-node set on trees with distinct sibling
                    tokens; emitted tokens equal plain greedy decoding of a
                    toy target model.
  adasd_stats       scipy's entropy and Jensen-Shannon distance; uniform,
                    one-hot, identical and disjoint rows in closed form.
  accept_adasd      reduces to accept_sample when nothing is relaxed and
                    nothing stops; d_eff from rows of known entropy; the
                    first emitted token follows the draft distribution where
                    JS <= tau (chi-square) and the target elsewhere.
  logits_to_probs   the fp64 softmax rounded to fp32: exact invariance to a
                    constant shift of the logits; a temperature of 1/2 equals
                    doubled logits; equal maxima give fl32(1 / k); two
                    logits give the logistic function; rows sum to 1 within
                    their rounding; the first emitted token follows the
                    target softmax (chi-square); its Philox equals the
                    independent implementation of the published definition
                    in synth bit for bit.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force=False):
    """Compile liboracle.so with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    # -ffp-contract=off: every fp32 step of the logits softmax rounds on its own
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-lm", "-o",
            _LIB + ".tmp"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_verify_attention.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                    i32, f64, i64, i32, P, P, P, i32]
            lib.oracle_gemm.argtypes = [P, P, i32, i32, i32, i32, P, P, i32]
            lib.oracle_accept_greedy.argtypes = [P, P, i32, i32, i32, P, P, i32]
            lib.oracle_accept_sample.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P, P, i32]
            lib.oracle_tree_attention.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                                  i32, f64, i64, i32, P, P, P, i32]
            lib.oracle_accept_tree_greedy.argtypes = [P, P, P, i32, i32, i32, P, P, P, i32]
            lib.oracle_accept_tree_sample.argtypes = [P, P, P, P, P, P, i32, i32, i32, P, P, P, P, P, i32]
            lib.oracle_logits_to_probs.argtypes = [P, P, ctypes.c_float, ctypes.c_uint64, i32, i32, i32,
                                                   P, P, P, P, i32]
            lib.oracle_logits_row_stats.argtypes = [P, P, ctypes.c_float, i32, i32, i32, P, P, i32]
            lib.oracle_adasd_stats.argtypes = [P, P, i32, i32, i32, P, P, i32]
            lib.oracle_accept_adasd.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, i32, i32, i32,
                                                P, P, P, P, P, P, i32]
            for f in ("oracle_verify_attention", "oracle_gemm", "oracle_accept_greedy",
                      "oracle_accept_sample", "oracle_max_threads", "oracle_tree_attention",
                      "oracle_accept_tree_greedy", "oracle_accept_tree_sample", "oracle_logits_to_probs",
                      "oracle_logits_row_stats",
                      "oracle_adasd_stats", "oracle_accept_adasd"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads():
    return _load().oracle_max_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def verify_attention(q, k_pages, v_pages, block_table, kv_len, D, Hkv, G, head_dim,
                     page_size, softmax_scale=None, rows=None, threads=0):
    """fp64 verify attention.

    q: uint16 bf16 bits [B, 1+D, Hkv*G, d]; k_pages/v_pages: uint16
    [P, page, Hkv, d]; block_table int32 [B, max_pages]; kv_len int32 [B].
    rows: optional int array [n, 4] of (b, i, h, g).  Returns (out, lse):
    full shapes [B, 1+D, Hq, d] / [B, 1+D, Hq], or [n, d] / [n].
    """
    lib = _load()
    q, k_pages, v_pages = (_c(a, np.uint16) for a in (q, k_pages, v_pages))
    block_table = _c(block_table, np.int32)
    kv_len = _c(kv_len, np.int32)
    B = kv_len.shape[0]
    Hq = Hkv * G
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(head_dim)
    P = k_pages.shape[0]
    if rows is not None:
        rows = _c(rows, np.int32).reshape(-1, 4)
        n = rows.shape[0]
        out = np.empty((n, head_dim), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
    else:
        n = 0
        out = np.empty((B, 1 + D, Hq, head_dim), dtype=np.float64)
        lse = np.empty((B, 1 + D, Hq), dtype=np.float64)
    rc = lib.oracle_verify_attention(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                     block_table.shape[1], _ptr(kv_len), B, D, Hkv, G, head_dim,
                                     page_size, float(softmax_scale), P, n, _ptr(rows), _ptr(out),
                                     _ptr(lse), int(threads))
    if rc:
        raise ValueError(f"oracle_verify_attention failed: {rc}")
    return out, lse


def gemm(x, w, samples=None, threads=0):
    """fp64 y = x @ w.T for bf16 bits x [M, K], w [N, K]; samples [n, 2]."""
    lib = _load()
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    if samples is not None:
        samples = _c(samples, np.int32).reshape(-1, 2)
        y = np.empty((samples.shape[0],), dtype=np.float64)
        n = samples.shape[0]
    else:
        y = np.empty((M, N), dtype=np.float64)
        n = 0
    rc = lib.oracle_gemm(_ptr(x), _ptr(w), M, N, K, n, _ptr(samples), _ptr(y), int(threads))
    if rc:
        raise ValueError(f"oracle_gemm failed: {rc}")
    return y


def accept_greedy(p, draft, threads=0):
    """Greedy prefix acceptance: returns (n_accepted [B], token [B]) int32."""
    lib = _load()
    p = _c(p, np.float32)
    draft = _c(draft, np.int32)
    B, D1, V = p.shape
    D = D1 - 1
    n_acc = np.empty((B,), np.int32)
    tok = np.empty((B,), np.int32)
    rc = lib.oracle_accept_greedy(_ptr(p), _ptr(draft), B, D, V, _ptr(n_acc), _ptr(tok),
                                  int(threads))
    if rc:
        raise ValueError(f"oracle_accept_greedy failed: {rc}")
    return n_acc, tok


def accept_sample(p, q, draft, u_acc, u_res, threads=0):
    """Stochastic acceptance: returns (n_accepted, token, margin, fallback)."""
    lib = _load()
    p, q = _c(p, np.float32), _c(q, np.float32)
    draft = _c(draft, np.int32)
    u_acc, u_res = _c(u_acc, np.float32), _c(u_res, np.float32)
    B, D1, V = p.shape
    D = D1 - 1
    n_acc = np.empty((B,), np.int32)
    tok = np.empty((B,), np.int32)
    margin = np.empty((B,), np.float64)
    fb = np.empty((B,), np.int32)
    rc = lib.oracle_accept_sample(_ptr(p), _ptr(q), _ptr(draft), _ptr(u_acc), _ptr(u_res),
                                  B, D, V, _ptr(n_acc), _ptr(tok), _ptr(margin), _ptr(fb),
                                  int(threads))
    if rc:
        raise ValueError(f"oracle_accept_sample failed: {rc}")
    return n_acc, tok, margin, fb


def tree_attention(q, k_pages, v_pages, block_table, kv_len, parent, D, Hkv, G, head_dim,
                   page_size, softmax_scale=None, rows=None, threads=0):
    """fp64 tree verify attention (reading R7).  As verify_attention, plus
    parent int32 [B, 1+D] (parent[:, 0] = -1, 0 <= parent[b, k] < k)."""
    lib = _load()
    q, k_pages, v_pages = (_c(a, np.uint16) for a in (q, k_pages, v_pages))
    block_table = _c(block_table, np.int32)
    kv_len = _c(kv_len, np.int32)
    parent = _c(parent, np.int32)
    B = kv_len.shape[0]
    Hq = Hkv * G
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(head_dim)
    P = k_pages.shape[0]
    if rows is not None:
        rows = _c(rows, np.int32).reshape(-1, 4)
        n = rows.shape[0]
        out = np.empty((n, head_dim), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
    else:
        n = 0
        out = np.empty((B, 1 + D, Hq, head_dim), dtype=np.float64)
        lse = np.empty((B, 1 + D, Hq), dtype=np.float64)
    rc = lib.oracle_tree_attention(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                   block_table.shape[1], _ptr(kv_len), _ptr(parent), B, D, Hkv, G,
                                   head_dim, page_size, float(softmax_scale), P, n, _ptr(rows),
                                   _ptr(out), _ptr(lse), int(threads))
    if rc:
        raise ValueError(f"oracle_tree_attention failed: {rc}")
    return out, lse


def accept_tree_greedy(p, tokens, parent, threads=0):
    """Greedy tree acceptance (reading R8): p float32 [B, 1+D, V], tokens and
    parent int32 [B, 1+D].  Returns (n_accepted, token, path [B, D])."""
    lib = _load()
    p = _c(p, np.float32)
    tokens = _c(tokens, np.int32)
    parent = _c(parent, np.int32)
    B, T, V = p.shape
    D = T - 1
    n = np.empty(B, np.int32)
    t = np.empty(B, np.int32)
    path = np.empty((B, max(D, 1)), np.int32)
    rc = lib.oracle_accept_tree_greedy(_ptr(p), _ptr(tokens), _ptr(parent), B, D, V, _ptr(n), _ptr(t),
                                       _ptr(path), int(threads))
    if rc:
        raise ValueError(f"oracle_accept_tree_greedy failed: {rc}")
    return n, t, path[:, :D]


def accept_tree_sample(p, q, tokens, parent, u_acc, u_res, threads=0):
    """Stochastic tree acceptance (reading R12): p, q float32 [B, 1+D, V]
    (q row k = the draft distribution node k's children were drawn from),
    tokens, parent int32 [B, 1+D], u_acc float32 [B, 1+D] (entry 0 unused),
    u_res float32 [B].  Returns (n_accepted, token, path [B, D], margin,
    flag)."""
    lib = _load()
    p, q = _c(p, np.float32), _c(q, np.float32)
    tokens, parent = _c(tokens, np.int32), _c(parent, np.int32)
    u_acc, u_res = _c(u_acc, np.float32), _c(u_res, np.float32)
    B, T, V = p.shape
    D = T - 1
    n = np.empty(B, np.int32)
    t = np.empty(B, np.int32)
    path = np.empty((B, max(D, 1)), np.int32)
    margin = np.empty(B, np.float64)
    flag = np.empty(B, np.int32)
    rc = lib.oracle_accept_tree_sample(_ptr(p), _ptr(q), _ptr(tokens), _ptr(parent), _ptr(u_acc), _ptr(u_res),
                                       B, D, V, _ptr(n), _ptr(t), _ptr(path), _ptr(margin), _ptr(flag),
                                       int(threads))
    if rc:
        raise ValueError(f"oracle_accept_tree_sample failed: {rc}")
    return n, t, path[:, :D], margin, flag


def logits_to_probs(zp, zq, temperature, seed, threads=0):
    """p, q (the fp64 softmax of logits / temperature rounded to fp32,
    reading R10) and the Philox uniforms u_acc, u_res (reading R11)."""
    lib = _load()
    zp = _c(zp, np.float32)
    zq = _c(zq, np.float32)
    B, T, V = zp.shape
    D = T - 1
    p = np.empty_like(zp)
    q = np.empty((B, D, V), np.float32)
    u_acc = np.empty((B, max(D, 1)), np.float32)
    u_res = np.empty(B, np.float32)
    rc = lib.oracle_logits_to_probs(_ptr(zp), _ptr(zq), float(temperature), int(seed), B, D, V, _ptr(p),
                                    _ptr(q), _ptr(u_acc), _ptr(u_res), int(threads))
    if rc:
        raise ValueError(f"oracle_logits_to_probs failed: {rc}")
    return p, q, np.ascontiguousarray(u_acc[:, :D]), u_res


def logits_row_stats(zp, zq, temperature, threads=0):
    """(m, Z) of reading R10 for every row: m [B, 2D + 1] fp32 (the row
    maximum) and Z [B, 2D + 1] fp64 (sum of exp((z - m) / T)), row k <= D
    being target row k and row k > D draft row k - D - 1; rows without a
    softmax (NaN, +inf or no finite entry) give (0, +inf)."""
    lib = _load()
    zp = _c(zp, np.float32)
    zq = _c(zq, np.float32)
    B, T, V = zp.shape
    D = T - 1
    m = np.empty((B, 2 * D + 1), np.float32)
    Z = np.empty((B, 2 * D + 1), np.float64)
    rc = lib.oracle_logits_row_stats(_ptr(zp), _ptr(zq), float(temperature), B, D, V, _ptr(m), _ptr(Z),
                                     int(threads))
    if rc < 0:
        raise ValueError(f"oracle_logits_row_stats failed: {rc}")
    return m, Z


def accept_sample_logits(zp, zq, draft, temperature, seed, threads=0):
    """Stochastic acceptance from logits: logits_to_probs, then accept_sample."""
    p, q, u_acc, u_res = logits_to_probs(zp, zq, temperature, seed, threads)
    return accept_sample(p, q, draft, u_acc, u_res, threads)


def adasd_stats(p, q, threads=0):
    """Entropy H(q_i) and JS distance JS(p_i, q_i) of every draft position
    (readings R12, R13): two [B, D] fp64 arrays."""
    lib = _load()
    p = _c(p, np.float32)
    q = _c(q, np.float32)
    B, T, V = p.shape
    D = T - 1
    H = np.empty((B, D), np.float64)
    JS = np.empty((B, D), np.float64)
    rc = lib.oracle_adasd_stats(_ptr(p), _ptr(q), B, D, V, _ptr(H), _ptr(JS), int(threads))
    if rc:
        raise ValueError(f"oracle_adasd_stats failed: {rc}")
    return H, JS


def accept_adasd(p, q, draft, u_acc, u_res, tau_h, tau_js, threads=0):
    """AdaSD relaxed acceptance (readings R12-R14): n_accepted, token, d_eff,
    margin_u, margin_stat, fallback."""
    lib = _load()
    p = _c(p, np.float32)
    q = _c(q, np.float32)
    B, T, V = p.shape
    D = T - 1
    draft = _c(draft if D else np.zeros((B, 1), np.int32), np.int32)
    u_acc = _c(u_acc if D else np.zeros((B, 1), np.float32), np.float32)
    u_res = _c(u_res, np.float32)
    n = np.empty(B, np.int32)
    t = np.empty(B, np.int32)
    de = np.empty(B, np.int32)
    mu = np.empty(B, np.float64)
    ms = np.empty(B, np.float64)
    fb = np.empty(B, np.int32)
    rc = lib.oracle_accept_adasd(_ptr(p), _ptr(q), _ptr(draft), _ptr(u_acc), _ptr(u_res), float(tau_h),
                                 float(tau_js), B, D, V, _ptr(n), _ptr(t), _ptr(de), _ptr(mu), _ptr(ms),
                                 _ptr(fb), int(threads))
    if rc:
        raise ValueError(f"oracle_accept_adasd failed: {rc}")
    return n, t, de, mu, ms, fb
