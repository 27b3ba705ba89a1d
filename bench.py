#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verification step on one GB300.

One step = one pass of the whole verification path over one batch of
synthetic inputs resident in HBM:
  1. verify attention  B=64 sequences, L_b ~ U{4096..131072}, 64-token pages
                       in a random permutation, Hkv=8, G=8, head_dim=128, D=7
  2. verify GEMM       M = B(1+D) = 512, N = K = 6144 (bf16, fp32 accumulate)
  3. greedy accept     B=64, D=7, V=131072 fp32 target probabilities
  4. stochastic accept same shapes, draft probabilities at acceptance ~0.6
Headline metric: verified query tokens per second, B(1+D) / step time.

The default run also times, inside the same clock-sampled window, every
other workload of the verification step and prints them under "cases" of
the one JSON line: the throughput attention case (B=16, L=32768, D=15),
the large-group D-sweep (B=8, G=32, L=131072, D in {0,1,3,4,7,15}), the
GEMM M-sweep (8..4096 x 6144 x 6144), batched acceptance (B=256, D=7,
V=131072, alpha 0.4/0.6/0.8, greedy and stochastic), acceptance from
logits, AdaSD, draft-tree verification and the adaptive draft-length tiers.

Usage: python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl reference]
The path runs on one GPU; with WORLD_SIZE > 1 the GPU arm prints an
"unavailable" line and exits without using any GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "verified query-tokens/s (verify attention + verify GEMM + greedy and stochastic accept)"
UNIT = "tokens/s"
WORKLOAD = dict(B=64, D=7, Hkv=8, G=8, head_dim=128, page_size=64, L_lo=4096, L_hi=131072,
                V=131072, alpha=0.6, N=6144, K=6144, seed=2026)
CASE_GROUPS = ("attention", "dsweep", "gemm", "accept", "logits", "adasd", "tree", "adaptive")
# throughput attention: G(1+D) = 128 query rows per KV head, one full tile
THROUGHPUT_CASE = dict(B=16, Hkv=8, G=8, D=15, L=32768)
# large groups: the same cache verified at draft lengths around 128 / G - 1
DSWEEP_CASE = dict(B=8, Hkv=4, G=32, L=131072, Ds=(0, 1, 3, 4, 7, 15))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return dict(hbm_gbs=float(m["hbm_gbs"]), bf16_tflops=float(m["bf16_tflops"]),
                    bf16_tflops_sustained=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def attention_traffic_ratio():
    """DRAM bytes / algorithmic bytes of the attention kernel from the last
    ncu capture (profiles/verify_attention_traffic.json), or None if the
    kernel sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "verify_attention_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    csrc = os.path.join(ROOT, "speculative_decoding_verification_attention_gb300", "csrc")
    src = "".join(open(os.path.join(csrc, n)).read() for n in ("attention.cu", "attn_schedule.h", "common.cuh"))
    if hashlib.sha256(src.encode()).hexdigest() != rec.get("source_sha256"):
        return None
    return float(rec["ratio"]), rec.get("case", "")


# ---------------------------------------------------------------- workload
class Workload:
    """Device-resident inputs of one verification step."""

    def __init__(self, device, seed=WORKLOAD["seed"]):
        import torch
        w = WORKLOAD
        self.B, self.D, self.V = w["B"], w["D"], w["V"]
        self.kv_len_host = synth.full_step_kv_lengths(seed, w["B"], w["L_lo"], w["L_hi"])
        self.attn = synth.attention_inputs_device(seed + 1, w["B"], w["Hkv"], w["G"],
                                                  w["head_dim"], w["D"], self.kv_len_host,
                                                  page_size=w["page_size"], device=device)
        g = torch.Generator(device=device)
        g.manual_seed(seed + 2)
        M = w["B"] * (1 + w["D"])
        self.M = M
        self.x = torch.randn((M, w["K"]), generator=g, device=device).to(torch.bfloat16)
        self.w = (torch.randn((w["N"], w["K"]), generator=g, device=device) * 0.02).to(torch.bfloat16)
        # acceptance inputs: fp32 softmax of N(0, 3^2) target logits; draft
        # logits = target + N(0, sigma^2) with sigma tuned for alpha
        sigma, _ = synth.tune_sigma_for_alpha(w["alpha"], w["V"], rows=8, target_std=3.0)
        self.sigma = sigma
        t = torch.randn((w["B"], w["D"] + 1, w["V"]), generator=g, device=device) * 3.0
        dl = t[:, :w["D"], :] + torch.randn((w["B"], w["D"], w["V"]), generator=g, device=device) * sigma
        self.p = torch.softmax(t.double(), dim=-1).float()
        self.q = torch.softmax(dl.double(), dim=-1).float()
        del t, dl
        u_acc, u_res = synth.acceptance_uniforms(seed + 3, w["B"], w["D"])
        b = np.arange(w["B"], dtype=np.uint64)
        i = np.arange(w["D"], dtype=np.uint64)
        ud = synth.philox_uniform(seed + 3, b[:, None], i[None, :], synth.STREAM_DRAFT)
        q_host = self.q.cpu().numpy()
        self.draft_sample = torch.from_numpy(synth.draw_from_rows(q_host, ud)).to(device)
        self.draft_greedy = torch.from_numpy(np.argmax(q_host, axis=-1).astype(np.int32)).to(device)
        del q_host
        self.u_acc = torch.from_numpy(u_acc).to(device)
        self.u_res = torch.from_numpy(u_res).to(device)
        self.sum_L = int(self.kv_len_host.astype(np.int64).sum())

    # algorithmic bytes / flops per launch
    def attention_bytes(self):
        w = WORKLOAD
        kv = 2 * self.sum_L * w["Hkv"] * w["head_dim"] * 2
        q = self.B * (1 + self.D) * w["Hkv"] * w["G"] * w["head_dim"] * 2
        o = self.B * (1 + self.D) * w["Hkv"] * w["G"] * (w["head_dim"] + 1) * 4
        return kv + q + o

    def attention_flops(self):
        w = WORKLOAD
        rows = (1 + self.D) * w["G"]
        return 4 * self.sum_L * w["Hkv"] * rows * w["head_dim"]

    def gemm_flops(self):
        return 2 * self.M * WORKLOAD["N"] * WORKLOAD["K"]

    def gemm_bytes(self):
        return 2 * (self.M * WORKLOAD["K"] + WORKLOAD["N"] * WORKLOAD["K"] + self.M * WORKLOAD["N"])


def accept_bytes(n_acc_greedy, n_acc_sample, B, D, V):
    greedy = int((np.asarray(n_acc_greedy) + 1).sum()) * V * 4
    rows = np.where(np.asarray(n_acc_sample) < D, 2, 1)
    sample = int(rows.sum()) * V * 4 + B * D * 16
    return greedy, sample


# ---------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, out_path):
        self.path = out_path
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, device_index=0):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9 or parts[0] != str(device_index):
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- GPU arm
def run_step(sv, wl, ws, outs, ev=None):
    """Enqueue one verification step; ev: optional list of 5 events."""
    a = wl.attn
    if ev: ev[0].record()
    sv.verify_attention(a.q, a.k_pages, a.v_pages, a.block_table, a.kv_len, wl.D, WORKLOAD["Hkv"],
                        WORKLOAD["G"], out=outs["o"], lse=outs["lse"], workspace=ws["attn"])
    if ev: ev[1].record()
    sv.verify_gemm(wl.x, wl.w, y=outs["y"], workspace=ws["gemm"])
    if ev: ev[2].record()
    sv.accept_greedy(wl.p, wl.draft_greedy, n_accepted=outs["ng"], token=outs["tg"])
    if ev: ev[3].record()
    sv.accept_sample(wl.p, wl.q, wl.draft_sample, wl.u_acc, wl.u_res, n_accepted=outs["ns"],
                     token=outs["ts"], workspace=ws["accept"])
    if ev: ev[4].record()


def gpu_arm(args):
    import torch
    from speculative_decoding_verification_attention_gb300 import _build
    import speculative_decoding_verification_attention_gb300 as sv

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sv.library()
    wl = Workload(dev)
    w = WORKLOAD
    Hq = w["Hkv"] * w["G"]
    outs = dict(o=torch.empty((wl.B, wl.D + 1, Hq, w["head_dim"]), device=dev),
                lse=torch.empty((wl.B, wl.D + 1, Hq), device=dev),
                y=torch.empty((wl.M, w["N"]), dtype=torch.bfloat16, device=dev),
                ng=torch.empty(wl.B, dtype=torch.int32, device=dev),
                tg=torch.empty(wl.B, dtype=torch.int32, device=dev),
                ns=torch.empty(wl.B, dtype=torch.int32, device=dev),
                ts=torch.empty(wl.B, dtype=torch.int32, device=dev))
    max_len = wl.attn.block_table.shape[1] * w["page_size"]
    ws = dict(attn=torch.empty(max(256, sv.attention_workspace_size(wl.B, wl.D, w["Hkv"], w["G"],
                                                                        w["head_dim"], max_len)),
                               dtype=torch.uint8, device=dev),
              gemm=torch.zeros(max(256, sv.gemm_workspace_size(wl.x.shape[0], wl.w.shape[0],
                                                               wl.x.shape[1])),
                               dtype=torch.uint8, device=dev),
              accept=torch.zeros(sv.accept_sample_workspace_size(wl.B, wl.V), dtype=torch.uint8,
                                 device=dev))
    flush = L2Flush(dev)

    for i in range(args.warmup):
        flush(i)
        run_step(sv, wl, ws, outs)
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    clock_path = os.path.join(tempfile.gettempdir(), f"spec_clocks_{os.getpid()}.csv")
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    cases = []
    with ClockSampler(clock_path) as clk:
        for i in range(K):
            flush(i + 7)                         # evict L2 between steps (not timed)
            run_step(sv, wl, ws, outs, evs[i])
        torch.cuda.synchronize()
        # stretch the sampled window so a short run still yields samples
        time.sleep(max(0.0, 0.45 - (time.perf_counter() - t_wall)))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        per = np.array([[evs[i][k].elapsed_time(evs[i][k + 1]) for k in range(4)] for i in range(K)])
        if not args.no_cases:
            t_cases = time.perf_counter()
            cases = run_cases(args, CASE_GROUPS, dev, sv, flush, step=(wl, outs))
            wall_cases = time.perf_counter() - t_cases
    step_ms = per.sum(axis=1)
    ms_step = float(step_ms.mean())
    ng, ns = outs["ng"].cpu().numpy(), outs["ns"].cpu().numpy()
    g_bytes, s_bytes = accept_bytes(ng, ns, wl.B, wl.D, wl.V)

    # ------------------------------------------------------------- e2e
    e2e = e2e_arm(sv, wl, ws, outs, dev, args.e2e_steps) if args.e2e_steps > 0 else None

    pk = peaks()
    traffic = attention_traffic_ratio()
    attn_ms = float(per[:, 0].mean())
    gemm_ms = float(per[:, 1].mean())
    greedy_ms = float(per[:, 2].mean())
    sample_ms = float(per[:, 3].mean())
    attn_gbs = wl.attention_bytes() / (attn_ms * 1e-3) / 1e9
    gemm_tf = wl.gemm_flops() / (gemm_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": wl.B * (1 + wl.D) / (ms_step * 1e-3),
        "unit": UNIT, "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random bf16 KV/Q/W, softmax probabilities of random logits)",
        "config": {"workload": "full verify step: paged GQA attention B=64 L~U[4096,131072] "
                               "page=64 Hkv=8 G=8 d=128 D=7 + GEMM M=512 N=K=6144 + "
                               "greedy/stochastic accept B=64 D=7 V=131072 alpha~0.6",
                   "global_batch_sequences": wl.B, "draft_len": wl.D,
                   "tokens_per_step": wl.B * (1 + wl.D), "sum_kv_len": wl.sum_L,
                   "kv_cache_gb": 2 * wl.sum_L * w["Hkv"] * w["head_dim"] * 2 / 1e9,
                   "parallelism": "single GPU",
                   "l2": "flushed between steps (512 MB write + 256 MB read, untimed)",
                   "precision": "bf16 inputs, fp32 accumulate, P as bf16 hi+lo in P.V, fp32 attention "
                                "output; acceptance exact (fp64 products, fixed-point sums)"},
        "kernels": {
            "attention": {"ms": attn_ms, "GB_per_s": attn_gbs,
                          "frac_hbm": attn_gbs / pk["hbm_gbs"],
                          "algorithmic_bytes": wl.attention_bytes(),
                          "tflops": wl.attention_flops() / (attn_ms * 1e-3) / 1e12},
            "gemm_M512": {"ms": gemm_ms, "TFLOP_per_s": gemm_tf,
                          "frac_tensor": gemm_tf / pk["bf16_tflops"],
                          "peak": "bf16 burst (of measured)",
                          "GB_per_s": wl.gemm_bytes() / (gemm_ms * 1e-3) / 1e9},
            "accept_greedy": {"ms": greedy_ms, "algorithmic_bytes": g_bytes,
                              "GB_per_s": g_bytes / (greedy_ms * 1e-3) / 1e9,
                              "frac_hbm": g_bytes / (greedy_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "accepted_tokens_per_s": float((ng + 1).sum()) / (greedy_ms * 1e-3)},
            "accept_sample": {"ms": sample_ms, "algorithmic_bytes": s_bytes,
                              "GB_per_s": s_bytes / (sample_ms * 1e-3) / 1e9,
                              "frac_hbm": s_bytes / (sample_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "accepted_tokens_per_s": float((ns + 1).sum()) / (sample_ms * 1e-3),
                              "mean_AL": float((ns + 1).mean())},
        },
        "roofline": {"kernel": "verify_attention (main + partial merge)", "bound": "hbm",
                     "achieved": attn_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": attn_gbs / pk["hbm_gbs"],
                     "traffic": (None if traffic is None else traffic[0] * wl.attention_bytes()),
                     "traffic_note": ("DRAM read+write bytes per launch: the ratio to algorithmic bytes "
                                      "from an ncu capture of a smaller case (" + traffic[1] + "), "
                                      "scaled to this launch") if traffic is not None else
                                     "no capture of the current attention sources",
                     "peak_source": pk["source"] + " (copy bandwidth, of measured)"},
        # per step: attention main + merge, GEMM, greedy accept, and the
        # three stochastic-accept kernels (first rejection, stream, draw)
        "gpu_launches": 7 * K,
        "wall_s_timed_region": wall,
        "clocks": clk.summary(dev.index or 0),
    }
    if cases:
        line["cases"] = cases
        line["cases_note"] = ("each case timed alone with CUDA events on its launching stream after "
                              f"{args.warmup} warm-up launches, mean of {case_steps(args)}; L2 flushed "
                              "between launches where the inputs fit in it; the clock record covers "
                              f"the headline step and all cases ({wall_cases:.1f} s)")
    if e2e is not None:
        line["e2e"] = e2e
    return line


def e2e_arm(sv, wl, ws, outs, dev, steps):
    """Same step through the public API with per-step inputs in pinned host
    memory: H2D of queries, page table, lengths, GEMM input, target/draft
    probabilities, drafts and uniforms; D2H of the accepted counts and
    tokens.  The KV cache and the weights stay resident (model state).

    The device inputs are double-buffered: step s + 1's inputs are uploaded
    on a copy stream while step s computes, as a serving loop would do.
    Every step's uploads and result read lie inside the timed region (the
    first upload starts after the start event, the last read ends before
    the stop event)."""
    import torch
    a = wl.attn
    host = {}
    for name, t in [("q", a.q), ("bt", a.block_table), ("kv", a.kv_len), ("x", wl.x),
                    ("p", wl.p), ("qd", wl.q), ("ds", wl.draft_sample), ("dg", wl.draft_greedy),
                    ("ua", wl.u_acc), ("ur", wl.u_res)]:
        host[name] = t.cpu().pin_memory()
    dst = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    res = torch.empty((4, wl.B), dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = res.numel() * res.element_size()
    Hkv, G = WORKLOAD["Hkv"], WORKLOAD["G"]
    compute = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]   # step's inputs landed in buffer i
    free = [torch.cuda.Event() for _ in range(2)]    # compute is done reading buffer i

    def upload(step):
        i = step % 2
        if step >= 2:
            copy.wait_event(free[i])
        with torch.cuda.stream(copy):
            for k in host:
                dst[i][k].copy_(host[k], non_blocking=True)
        ready[i].record(copy)

    def run(step):
        i = step % 2
        d = dst[i]
        compute.wait_event(ready[i])
        sv.verify_attention(d["q"], a.k_pages, a.v_pages, d["bt"], d["kv"], wl.D, Hkv, G,
                            out=outs["o"], lse=outs["lse"], workspace=ws["attn"])
        sv.verify_gemm(d["x"], wl.w, y=outs["y"], workspace=ws["gemm"])
        sv.accept_greedy(d["p"], d["dg"], n_accepted=outs["ng"], token=outs["tg"])
        sv.accept_sample(d["p"], d["qd"], d["ds"], d["ua"], d["ur"],
                         n_accepted=outs["ns"], token=outs["ts"], workspace=ws["accept"])
        free[i].record(compute)
        res[0].copy_(outs["ng"], non_blocking=True)
        res[1].copy_(outs["tg"], non_blocking=True)
        res[2].copy_(outs["ns"], non_blocking=True)
        res[3].copy_(outs["ts"], non_blocking=True)

    def loop(n, start_event=None):
        if start_event is not None:
            copy.wait_event(start_event)
        upload(0)
        for s in range(n):
            if s + 1 < n:
                upload(s + 1)
            run(s)

    loop(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    loop(steps, e0)
    e1.record(compute)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": wl.B * (1 + wl.D) / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "note": "KV cache and GEMM weights resident; per-step inputs copied from pinned host, "
                    "step s+1's upload (copy stream) overlapping step s's compute"}


# ------------------------------------------------------ single-kernel cases
class L2Flush:
    """Evicts L2 between timed launches (untimed): writes a 512 MB buffer
    (> the 129 MB L2), then reads a 256 MB one so that the lines left in L2
    are clean -- otherwise the next kernel would pay for writing back the
    flush's own dirty lines."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self, i):
        self.w.fill_(i & 0xFF)
        self.r.sum()


def time_launches(fn, warmup, steps, flush=None):
    """Mean device time (ms) of fn() over `steps` launches after `warmup`,
    flushing L2 between launches when a flush buffer is given."""
    import torch
    for i in range(warmup):
        if flush is not None:
            flush(i)
        fn()
    torch.cuda.synchronize()
    ts = []
    for i in range(steps):
        if flush is not None:
            flush(i + 3)
        # keep the GPU busy (~0.5 ms, outside the timed events) while the host
        # enqueues the launch, so the events measure device time only
        torch.cuda._sleep(1_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        ts.append((e0, e1))
        torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ts]))


def case_steps(args):
    return max(3, min(args.steps, 10))


def device_drafts(q, seed):
    """Draft tokens of the acceptance inputs, synthesised on the device:
    draft i of sequence b is drawn from q[b, i] by inverse CDF (fp64 running
    sum) with the Philox uniform of counter (b, i, draft stream) -- sample
    mode -- or is argmax q[b, i], lowest index on ties -- greedy mode."""
    import torch
    B, D, V = q.shape
    ud = synth.philox_uniform(seed, np.arange(B, dtype=np.uint64)[:, None],
                              np.arange(D, dtype=np.uint64)[None, :], synth.STREAM_DRAFT)
    u = torch.from_numpy(np.asarray(ud, dtype=np.float64)).to(q.device)
    ds = torch.empty((B, D), dtype=torch.int32, device=q.device)
    for s in range(0, B, 16):
        c = torch.cumsum(q[s:s + 16].double(), -1)
        t = (u[s:s + 16, :, None] * c[:, :, -1:]).contiguous()
        ds[s:s + 16] = torch.searchsorted(c, t, right=True).squeeze(-1).clamp_max(V - 1).int()
        del c, t
    dg = torch.argmax(q, -1).int()
    return ds, dg


def device_probs(B, D, V, sigma, seed, dev, target_std=3.0):
    """fp32 target / draft probabilities: softmax (in fp64) of N(0, 3^2)
    target logits and of the target logits plus N(0, sigma^2) noise."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    p = torch.empty((B, D + 1, V), device=dev)
    q = torch.empty((B, D, V), device=dev)
    for s in range(0, B, 32):
        n = min(32, B - s)
        t = torch.randn((n, D + 1, V), generator=g, device=dev) * target_std
        p[s:s + n] = torch.softmax(t.double(), -1).float()
        q[s:s + n] = torch.softmax((t[:, :D] + torch.randn((n, D, V), generator=g, device=dev)
                                    * sigma).double(), -1).float()
        del t
    return p, q


def attention_record(name, B, Hkv, G, D, sumL, ms, pk, d=128):
    by = 2 * sumL * Hkv * d * 2 + B * (D + 1) * Hkv * G * (d * 2 + (d + 1) * 4)
    fl = 4 * sumL * Hkv * G * (1 + D) * d
    m_tiles = (G * (1 + D) + 127) // 128
    fl_pad = 4 * sumL * Hkv * 128 * m_tiles * d
    gbs = by / (ms * 1e-3) / 1e9
    tf_pad = fl_pad / (ms * 1e-3) / 1e12
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    t_tc = fl_pad / (pk["bf16_tflops"] * 1e12)
    return {"case": name, "kernel": "verify_attention", "B": B, "Hkv": Hkv, "G": G, "D": D,
            "G(1+D)": G * (1 + D), "m_tiles_per_kv_head": m_tiles, "ms": ms,
            "query_tokens_per_s": B * (D + 1) / (ms * 1e-3), "algorithmic_bytes": by,
            "GB_per_s": gbs, "frac_hbm": gbs / pk["hbm_gbs"],
            "TFLOP_per_s": fl / (ms * 1e-3) / 1e12, "padded_TFLOP_per_s": tf_pad,
            "frac_tensor_padded": tf_pad / pk["bf16_tflops"],
            "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "frac": (t_hbm if t_hbm >= t_tc else t_tc) / (ms * 1e-3)}


def run_cases(args, groups, dev, sv, flush, step=None):
    """Time the secondary workloads of the verification step; returns one
    record per case.  step: (Workload, outputs) of the headline step, whose
    resident inputs the tree case reuses."""
    import torch
    pk = peaks()
    W, S = args.warmup, case_steps(args)
    recs = []

    if "attention" in groups:
        # throughput regime: G(1+D) = 128, one full query tile per KV head
        c = THROUGHPUT_CASE
        B, Hkv, G, D, L = c["B"], c["Hkv"], c["G"], c["D"], c["L"]
        inp = synth.attention_inputs_device(11, B, Hkv, G, 128, D, L, page_size=64, device=dev)
        out = torch.empty((B, D + 1, Hkv * G, 128), device=dev)
        lse = torch.empty((B, D + 1, Hkv * G), device=dev)
        wsa = torch.empty(sv.attention_workspace_size(B, D, Hkv, G, 128, L), dtype=torch.uint8, device=dev)
        ms = time_launches(lambda: sv.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                                       inp.kv_len, D, Hkv, G, out=out, lse=lse, workspace=wsa),
                           W, S)   # 2.1 GB of K/V, larger than L2
        recs.append(attention_record(f"attention B{B} Hkv{Hkv} G{G} L{L} D{D}", B, Hkv, G, D, B * L, ms, pk))
        del inp, out, lse, wsa
        torch.cuda.empty_cache()

    if "dsweep" in groups:
        # large groups: the same K/V cache (L = 131072 per sequence) verified
        # with D = 0, 1, 3, 4, 7, 15 (G(1+D) = 32 ... 512 query rows)
        c = DSWEEP_CASE
        B, Hkv, G, L = c["B"], c["Hkv"], c["G"], c["L"]
        inp = synth.attention_inputs_device(20, B, Hkv, G, 128, max(c["Ds"]), L, page_size=64, device=dev)
        for D in c["Ds"]:
            q = inp.q[:, :D + 1].contiguous()
            out = torch.empty((B, D + 1, Hkv * G, 128), device=dev)
            lse = torch.empty((B, D + 1, Hkv * G), device=dev)
            wsa = torch.empty(sv.attention_workspace_size(B, D, Hkv, G, 128, L), dtype=torch.uint8, device=dev)
            ms = time_launches(lambda: sv.verify_attention(q, inp.k_pages, inp.v_pages, inp.block_table,
                                                           inp.kv_len, D, Hkv, G, out=out, lse=lse,
                                                           workspace=wsa), W, S)
            recs.append(attention_record(f"attention D-sweep B{B} Hkv{Hkv} G{G} L{L} D{D}", B, Hkv, G, D,
                                         B * L, ms, pk))
            del q, out, lse, wsa
        del inp
        torch.cuda.empty_cache()

    if "gemm" in groups:
        N = K = 6144
        w = (torch.randn((N, K), device=dev) * 0.02).to(torch.bfloat16)
        ms_list = (args.gemm_m,) if args.gemm_m else (8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)
        for M in ms_list:
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsg = torch.zeros(max(256, sv.gemm_workspace_size(M, N, K)), dtype=torch.uint8, device=dev)
            ms = time_launches(lambda: sv.verify_gemm(x, w, y=y, workspace=wsg), W, S, flush)
            fl = 2 * M * N * K
            by = 2 * (M * K + N * K + M * N)
            tf = fl / (ms * 1e-3) / 1e12
            gbs = by / (ms * 1e-3) / 1e9
            tensor = fl / by > pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
            recs.append({"case": f"gemm M{M} N{N} K{K}", "kernel": "verify_gemm", "M": M, "ms": ms,
                         "TFLOP_per_s": tf, "frac_tensor": tf / pk["bf16_tflops"], "algorithmic_bytes": by,
                         "GB_per_s": gbs, "frac_hbm": gbs / pk["hbm_gbs"],
                         "bound": "tensor" if tensor else "hbm",
                         "frac": tf / pk["bf16_tflops"] if tensor else gbs / pk["hbm_gbs"]})
            del x, y, wsg
        del w
        torch.cuda.empty_cache()

    def accept_record(name, kernel, ms, n, by, **extra):
        gbs = by / (ms * 1e-3) / 1e9
        r = {"case": name, "kernel": kernel, "ms": ms,
             "accepted_tokens_per_s": float((n + 1).sum()) / (ms * 1e-3),
             "sequences_per_s": len(n) / (ms * 1e-3), "mean_AL": float((n + 1).mean()),
             "algorithmic_bytes": by, "GB_per_s": gbs, "frac_hbm": gbs / pk["hbm_gbs"], "bound": "hbm",
             "frac": gbs / pk["hbm_gbs"]}
        r.update(extra)
        return r

    if "accept" in groups:
        B, D, V = 256, 7, 131072
        for alpha in ((0.6,) if args.workload == "accept-one" else (0.4, 0.6, 0.8)):
            sigma, _ = synth.tune_sigma_for_alpha(alpha, V, rows=8, target_std=3.0)
            p, q = device_probs(B, D, V, sigma, int(alpha * 100), dev)
            ds, dg = device_drafts(q, 7)
            u_acc, u_res = synth.acceptance_uniforms(7, B, D)
            ua, ur = torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_res).to(dev)
            na, tk = torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev)
            ms_g = time_launches(lambda: sv.accept_greedy(p, dg, na, tk), W, S, flush)
            ng = na.cpu().numpy()
            wsa = torch.zeros(sv.accept_sample_workspace_size(B, V), dtype=torch.uint8, device=dev)
            ms_s = time_launches(lambda: sv.accept_sample(p, q, ds, ua, ur, na, tk, workspace=wsa), W, S, flush)
            ns = na.cpu().numpy()
            gb, sb = accept_bytes(ng, ns, B, D, V)
            recs.append(accept_record(f"accept greedy B{B} D{D} V{V} alpha{alpha}", "accept_greedy", ms_g, ng, gb,
                                      alpha=alpha))
            recs.append(accept_record(f"accept sample B{B} D{D} V{V} alpha{alpha}", "accept_sample", ms_s, ns, sb,
                                      alpha=alpha))
            del p, q, ds, dg, wsa
            torch.cuda.empty_cache()

    if "logits" in groups:
        # acceptance from logits: target logits N(0, 3^2), draft logits the
        # target's plus N(0, sigma^2) with sigma tuned to alpha = 0.6, T = 1
        B, D, V, T = (32 if args.workload == "logits-small" else 256), 7, 131072, 1.0
        sigma, _ = synth.tune_sigma_for_alpha(0.6, V, rows=8, target_std=3.0)
        g = torch.Generator(device=dev)
        g.manual_seed(60)
        zp = torch.randn((B, D + 1, V), generator=g, device=dev) * 3.0
        zq = (zp[:, :D] + torch.randn((B, D, V), generator=g, device=dev) * sigma).contiguous()
        ds, _ = device_drafts(torch.softmax(zq.double() / T, -1).float(), 7)
        na, tk = torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev)
        wsl = torch.empty(sv.accept_sample_logits_workspace_size(B, D, V), dtype=torch.uint8, device=dev)
        ms_f = time_launches(lambda: sv.accept_sample_logits(zp, zq, ds, T, 7, na, tk, workspace=wsl), W, S, flush)
        nf = na.cpu().numpy()
        rows_bytes = B * (2 * D + 1) * V * 4
        _, sb = accept_bytes(nf, nf, B, D, V)
        recs.append(accept_record(f"accept from logits B{B} D{D} V{V} T{T} alpha0.6", "accept_sample_logits",
                                  ms_f, nf, rows_bytes + sb, logit_bytes=rows_bytes))
        # the same decisions taken the unfused way: library fp32 softmax of
        # both tensors (written to HBM), then the probability-form kernels
        u_acc, u_res = synth.acceptance_uniforms(7, B, D)
        ua, ur = torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_res).to(dev)
        wsa = torch.empty(sv.accept_sample_workspace_size(B, V), dtype=torch.uint8, device=dev)
        ms_u = time_launches(lambda: sv.accept_sample(torch.softmax(zp, -1), torch.softmax(zq, -1), ds, ua, ur,
                                                      na, tk, workspace=wsa), W, S, flush)
        recs.append({"case": f"accept from logits, unfused (library softmax + accept_sample) B{B} D{D} V{V}",
                     "kernel": "torch.softmax x2 + accept_sample", "ms": ms_u, "speedup_of_fused": ms_u / ms_f})
        del zp, zq, ds, wsl, wsa
        torch.cuda.empty_cache()

    if "adasd" in groups:
        # AdaSD relaxed acceptance at alpha = 0.6; tau_H at the 90th
        # percentile of the draft entropies, tau_JS at the median distance
        B, D, V = (32 if args.workload == "adasd-small" else 256), 7, 131072
        sigma, _ = synth.tune_sigma_for_alpha(0.6, V, rows=8, target_std=3.0)
        p, q = device_probs(B, D, V, sigma, 61, dev)
        ds, _ = device_drafts(q, 8)
        u_acc, u_res = synth.acceptance_uniforms(8, B, D)
        ua, ur = torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_res).to(dev)
        na, tk = torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev)
        dl = torch.empty(B, dtype=torch.int32, device=dev)
        H = torch.empty((B, D), device=dev)
        JS = torch.empty((B, D), device=dev)
        wsd = torch.empty(sv.accept_adasd_workspace_size(B, D, V), dtype=torch.uint8, device=dev)
        sv.accept_adasd(p, q, ds, ua, ur, float("inf"), -1.0, na, tk, dl, H, JS, workspace=wsd)
        torch.cuda.synchronize()
        tau_h = float(torch.quantile(H.flatten(), 0.9))
        tau_js = float(torch.quantile(JS.flatten(), 0.5))
        ms_a = time_launches(lambda: sv.accept_adasd(p, q, ds, ua, ur, tau_h, tau_js, na, tk, dl, H, JS,
                                                     workspace=wsd), W, S, flush)
        n_a, d_a = na.cpu().numpy(), dl.cpu().numpy()
        _, sb = accept_bytes(n_a, np.where(n_a < d_a, 0, D), B, D, V)
        wsa = torch.empty(sv.accept_sample_workspace_size(B, V), dtype=torch.uint8, device=dev)
        ms_s = time_launches(lambda: sv.accept_sample(p, q, ds, ua, ur, na, tk, workspace=wsa), W, S, flush)
        n_s = na.cpu().numpy()
        recs.append(accept_record(f"accept AdaSD B{B} D{D} V{V} alpha0.6 tauH=p90 tauJS=p50", "accept_adasd",
                                  ms_a, n_a, B * D * 2 * V * 4 + sb, mean_d_eff=float(d_a.mean()),
                                  mean_AL_lossless=float((n_s + 1).mean()), ms_lossless=ms_s))
        del p, q, ds, wsd, wsa
        torch.cuda.empty_cache()

    if "tree" in groups:
        # tree verification over the headline step's resident inputs (B=64
        # paged sequences, L ~ U{4096..131072}, Hkv=8, G=8, d=128) with an
        # 8-node draft tree, against the chain on the same inputs
        B, Hkv, G, D = 64, 8, 8, 7
        if step is not None:
            inp = step[0].attn
            sumL = step[0].sum_L
        else:
            inp = synth.attention_inputs_device(51, B, Hkv, G, 128, D, synth.full_step_kv_lengths(50),
                                                page_size=64, device=dev)
            sumL = int(np.sum(inp.kv_len_host.astype(np.int64)))
        parent = torch.from_numpy(synth.tree_parents(3, B, D + 1, "wide")).to(dev)
        out = torch.empty((B, D + 1, Hkv * G, 128), device=dev)
        lse = torch.empty((B, D + 1, Hkv * G), device=dev)
        max_len = inp.block_table.shape[1] * 64
        wst = torch.empty(sv.tree_attention_workspace_size(B, D, Hkv, G, 128, max_len), dtype=torch.uint8, device=dev)
        ms = time_launches(lambda: sv.verify_tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                                            inp.kv_len, parent, D, Hkv, G, out=out, lse=lse,
                                                            workspace=wst), W, S)
        r = attention_record("tree attention B64 L~U[4096,131072] Hkv8 G8 D7 (8-node wide tree)", B, Hkv, G, D,
                             sumL, ms, pk)
        r["kernel"] = "verify_tree_attention"
        recs.append(r)
        wsc = torch.empty(sv.attention_workspace_size(B, D, Hkv, G, 128, max_len), dtype=torch.uint8, device=dev)
        ms_c = time_launches(lambda: sv.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                                         inp.kv_len, D, Hkv, G, out=out, lse=lse, workspace=wsc),
                             W, S)
        recs.append(attention_record("chain attention, same inputs as the tree case", B, Hkv, G, D, sumL, ms_c, pk))
        del parent, out, lse, wst, wsc
        if step is None:
            del inp
        torch.cuda.empty_cache()
        Bt, Vt = 256, 131072
        sigma, _ = synth.tune_sigma_for_alpha(0.6, Vt, rows=8, target_std=3.0)
        pt, _ = device_probs(Bt, D, Vt, sigma, 77, dev)
        par_h = synth.tree_parents(4, Bt, D + 1, "wide")
        am = torch.argmax(pt, -1).cpu().numpy()
        rng = np.random.default_rng(5)
        tok_h = rng.integers(0, Vt, size=(Bt, D + 1)).astype(np.int32)
        for k in range(1, D + 1):
            hit = rng.random(Bt) < 0.6
            tok_h[hit, k] = am[hit, par_h[hit, k]]
        tok, par = torch.from_numpy(tok_h).to(dev), torch.from_numpy(par_h).to(dev)
        na = torch.empty(Bt, dtype=torch.int32, device=dev)
        tk = torch.empty(Bt, dtype=torch.int32, device=dev)
        path = torch.empty((Bt, D), dtype=torch.int32, device=dev)
        ms_t = time_launches(lambda: sv.accept_tree_greedy(pt, tok, par, na, tk, path), W, S, flush)
        nacc = na.cpu().numpy().astype(np.int64)
        recs.append(accept_record(f"tree accept greedy B{Bt} D{D} V{Vt} wide tree", "accept_tree_greedy", ms_t,
                                  nacc, int(np.sum(nacc + 1)) * Vt * 4))
        del pt, tok, par
        torch.cuda.empty_cache()
        # stochastic tree acceptance on the same tree shape: a target and a
        # draft row per node (alpha ~ 0.6), each node's token drawn from the
        # draft row of its parent
        pt, qt = device_probs(Bt, D + 1, Vt, sigma, 78, dev)
        pt = pt[:, :D + 1].contiguous()
        bidx = torch.arange(Bt, device=dev)
        par_d = torch.from_numpy(par_h).to(dev).long()
        qsel = torch.stack([qt[bidx, par_d[:, k]] for k in range(1, D + 1)], 1)
        ds, _ = device_drafts(qsel, 79)
        del qsel
        tok = torch.zeros((Bt, D + 1), dtype=torch.int32, device=dev)
        tok[:, 1:] = ds
        ua, ur = synth.acceptance_uniforms(80, Bt, D + 1)
        ua, ur = torch.from_numpy(ua).to(dev), torch.from_numpy(ur).to(dev)
        par = torch.from_numpy(par_h).to(dev)
        ms_s = time_launches(lambda: sv.accept_tree_sample(pt, qt, tok, par, ua, ur, na, tk, path), W, S, flush)
        nacc = na.cpu().numpy().astype(np.int64)
        path_h = path.cpu().numpy()
        # algorithmic bytes: the distinct rows the rule must read -- a
        # node's p and q rows when one of its children is rejected there,
        # and p alone at the final node when none is.  Passes after the
        # first at a node re-read rows already read (on-chip or L2 traffic,
        # reported as passes per sequence, not counted as HBM bytes).
        kids = [[c for c in range(1, D + 1) if par_h[b, c] == v] for b in range(Bt) for v in range(D + 1)]
        passes = np.zeros(Bt, np.int64)
        rows = np.zeros(Bt, np.int64)
        for b in range(Bt):
            node = 0
            for d in range(int(nacc[b]) + 1):
                ch = kids[b * (D + 1) + node]
                if d < nacc[b]:
                    nxt = int(path_h[b, d])
                    rej = sum(1 for c in ch if c < nxt)
                    node = nxt
                else:
                    rej = len(ch)
                passes[b] += rej
                rows[b] += 2 if rej > 0 else (1 if d == nacc[b] else 0)
        by = int(rows.sum()) * Vt * 4
        recs.append(accept_record(f"tree accept sample B{Bt} D{D} V{Vt} wide tree alpha0.6", "accept_tree_sample",
                                  ms_s, nacc, by, row_passes_per_sequence=float(passes.mean()),
                                  rows_read_per_sequence=float(rows.mean())))
        del pt, qt, tok, par, ua, ur
        torch.cuda.empty_cache()

    if "adaptive" in groups:
        recs.extend(adaptive_cases(args, dev, sv))

    for r in recs:
        r["peak_source"] = pk["source"]
    return recs


def adaptive_cases(args, dev, sv):
    """One CUDA graph per draft-length tier of a verification step (verify
    attention B=8 L=4096 Hkv=8 G=8 d=128, the N=K=6144 linear layer at
    M=8(1+D), stochastic acceptance V=32768); host wall time per round,
    eager launches against graph replay, then a controller-driven run."""
    import torch
    from speculative_decoding_verification_attention_gb300.graphs import TierGraphs
    B, Hkv, G, L, V, N = 8, 8, 8, 4096, 32768, 6144
    tiers = (1, 3, 7)
    bufs = {}
    for D in tiers:
        a = synth.attention_inputs_device(90 + D, B, Hkv, G, 128, D, L, page_size=64, device=dev)
        p, q = device_probs(B, D, V, 0.5, 95 + D, dev, target_std=2.0)
        ds, _ = device_drafts(q, 95 + D)
        u_acc, u_res = synth.acceptance_uniforms(95 + D, B, D)
        M = B * (D + 1)
        bufs[D] = dict(
            a=a, out=torch.empty((B, D + 1, Hkv * G, 128), device=dev),
            wsa=torch.empty(sv.attention_workspace_size(B, D, Hkv, G, 128, L), dtype=torch.uint8, device=dev),
            x=torch.randn((M, N), device=dev).to(torch.bfloat16),
            w=(torch.randn((N, N), device=dev) * 0.02).to(torch.bfloat16),
            y=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
            wsg=torch.zeros(max(256, sv.gemm_workspace_size(M, N, N)), dtype=torch.uint8, device=dev),
            acc=dict(p=p, q=q, draft=ds, u_acc=torch.from_numpy(u_acc).to(dev), u_res=torch.from_numpy(u_res).to(dev)),
            na=torch.empty(B, dtype=torch.int32, device=dev), tk=torch.empty(B, dtype=torch.int32, device=dev),
            wss=torch.empty(sv.accept_sample_workspace_size(B, V), dtype=torch.uint8, device=dev))

    def step(D):
        s = bufs[D]
        a, c = s["a"], s["acc"]
        sv.verify_attention(a.q, a.k_pages, a.v_pages, a.block_table, a.kv_len, D, Hkv, G, out=s["out"],
                            workspace=s["wsa"])
        sv.verify_gemm(s["x"], s["w"], y=s["y"], workspace=s["wsg"])
        sv.accept_sample(c["p"], c["q"], c["draft"], c["u_acc"], c["u_res"], s["na"], s["tk"],
                         workspace=s["wss"])

    graphs = TierGraphs(step, tiers)

    def wall(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
            torch.cuda.synchronize()   # a round ends when its acceptance is known
        return (time.perf_counter() - t0) / n * 1e3

    recs = []
    for D in tiers:
        n = max(10, case_steps(args) * 5)
        ms_e = wall(lambda: step(D), n)
        ms_g = wall(lambda: graphs.replay(D), n)
        recs.append({"case": f"adaptive tier D={D}: round B{B} L{L} V{V} (attention + GEMM + sample accept)",
                     "kernel": "tier graph", "D": D, "ms_eager_wall": ms_e, "ms_graph_wall": ms_g,
                     "ms": ms_g, "verified_tokens_per_s_graph": B * (D + 1) / (ms_g * 1e-3),
                     "timing": "host wall clock per round, synchronised"})
    # a controller-driven run: acceptance drifts from low to high and back
    ctl = sv.AdaptiveDraftLength(tiers, beta=0.7)
    rng = np.random.default_rng(0)
    alphas = np.concatenate([np.full(40, 0.2), np.full(40, 0.9), np.full(40, 0.4)])
    used, acc_tok = [], 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for al in alphas:
        D = ctl.draft_len
        used.append(D)
        graphs.replay(D)
        torch.cuda.synchronize()
        n_acc = np.minimum(rng.geometric(1.0 - al, size=B) - 1, D)   # synthetic acceptance
        acc_tok += int(np.sum(n_acc + 1))
        ctl.update(n_acc.astype(np.int32))
    dt = time.perf_counter() - t0
    recs.append({"case": "adaptive controller over 120 rounds (acceptance 0.2 -> 0.9 -> 0.4)",
                 "kernel": "tier graphs + controller", "ms": dt / len(alphas) * 1e3,
                 "rounds_per_tier": {str(D): int(np.sum(np.asarray(used) == D)) for D in tiers},
                 "accepted_tokens_per_s": acc_tok / dt, "timing": "host wall clock"})
    del bufs, graphs
    torch.cuda.empty_cache()
    return recs


def case_lines(args):
    """--workload other than step: one JSON line per case (no headline)."""
    import torch
    from speculative_decoding_verification_attention_gb300 import _build
    import speculative_decoding_verification_attention_gb300 as sv
    _build.build()
    sv.library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    wk = args.workload
    if wk == "all":
        groups = CASE_GROUPS
    elif wk in CASE_GROUPS:
        groups = (wk,)
    elif wk in ("accept-one", "logits-small", "adasd-small"):
        groups = (wk.split("-")[0],)
    else:
        groups = ()
    recs = run_cases(args, groups, dev, sv, flush) if groups else []
    pk = peaks()
    # profiling cases: small inputs for ncu captures (a few hundred MB)
    small = {"attention-small": (4, 8, 8, 7, 32768, 5),
             "attention-small-d15": (4, 8, 8, 15, 32768, 6),
             "attention-largeg-small": (1, 4, 32, 15, 131072, 35)}
    if wk in small:
        B, Hkv, G, D, L, seed = small[wk]
        inp = synth.attention_inputs_device(seed, B, Hkv, G, 128, D, L, page_size=64, device=dev)
        out = torch.empty((B, D + 1, Hkv * G, 128), device=dev)
        lse = torch.empty((B, D + 1, Hkv * G), device=dev)
        wsa = torch.empty(sv.attention_workspace_size(B, D, Hkv, G, 128, L), dtype=torch.uint8, device=dev)
        ms = time_launches(lambda: sv.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                                       inp.kv_len, D, Hkv, G, out=out, lse=lse, workspace=wsa),
                           args.warmup, args.steps)
        recs.append(attention_record(f"{wk} B{B} Hkv{Hkv} G{G} L{L} D{D} (profiling)", B, Hkv, G, D, B * L, ms, pk))
    for r in recs:
        r["peak_source"] = pk["source"]
        print(json.dumps(r), flush=True)


# ---------------------------------------------------------------- CPU arm
def cpu_sample_time(threads=0, budget_s=12.0):
    """Time the fp64 oracle on a bounded sample of one step and extrapolate
    to the whole step.  Returns (extrapolated seconds per step, seconds the
    sample actually took, description, threads).

    The sample: whole (b, h) attention units of a 16384-key sequence (all 64
    query rows) until about 70% of the budget is spent, 4 of the 512 GEMM
    rows, and 16 of the 64 sequences of acceptance (both modes); each part is
    scaled linearly (keys x heads, rows, sequences) to the full step.
    """
    import oracle
    w = WORKLOAD
    kv = synth.full_step_kv_lengths(WORKLOAD["seed"], w["B"], w["L_lo"], w["L_hi"])
    sum_L = int(kv.astype(np.int64).sum())
    nthreads = oracle.max_threads() if threads <= 0 else threads
    L = 16384
    inp = synth.attention_inputs(1, 1, 1, w["G"], w["head_dim"], w["D"], [L], page_size=64)
    n_units = 0
    t_start = time.perf_counter()
    t0 = time.perf_counter()
    while n_units < 1 or (time.perf_counter() - t0 < 0.7 * budget_s and n_units < 64):
        oracle.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                w["D"], 1, w["G"], w["head_dim"], 64, threads=threads)
        n_units += 1
    t_attn = (time.perf_counter() - t0) / (n_units * L) * sum_L * w["Hkv"]
    M = w["B"] * (1 + w["D"])
    x, wt = synth.gemm_inputs(2, 4, w["N"], w["K"])
    t0 = time.perf_counter()
    oracle.gemm(x, wt, threads=threads)
    t_gemm = (time.perf_counter() - t0) / 4 * M
    acc = synth.accept_inputs(3, 16, w["D"], w["V"], target_std=3.0, draft_noise=1.0, mode="both")
    t0 = time.perf_counter()
    oracle.accept_greedy(acc["p"], acc["draft_greedy"], threads=threads)
    oracle.accept_sample(acc["p"], acc["q"], acc["draft_sample"], acc["u_acc"], acc["u_res"],
                         threads=threads)
    t_acc = (time.perf_counter() - t0) / 16 * w["B"]
    sampled = time.perf_counter() - t_start
    total = t_attn + t_gemm + t_acc
    desc = (f"fp64 oracle on {n_units} attention unit(s) of {L} keys x 64 rows (scaled by keys "
            f"to sum L={sum_L} over {w['Hkv']} KV heads), 4 of {M} GEMM rows, 16 of {w['B']} "
            f"sequences of greedy+stochastic acceptance; each part's time extrapolated linearly "
            f"to one whole step")
    return total, sampled, desc, nthreads


def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    times, sampled = [], []
    desc, nthreads = "", 0
    for i in range(args.warmup + args.steps):
        t, s, desc, nthreads = cpu_sample_time(budget_s=args.cpu_budget_s)
        if i >= args.warmup:
            times.append(t)
            sampled.append(s)
    ms = 1e3 * float(np.mean(times))
    tokens = WORKLOAD["B"] * (1 + WORKLOAD["D"])
    v = tokens / (ms * 1e-3)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_kind": "extrapolated: each step runs a bounded sample of the step on the host "
                                "cores and scales each part's time linearly to the whole step",
            "sampled_s_per_step": float(np.mean(sampled)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "full verify step (same as the GPU arm), evaluated by the "
                                   "fp64 CPU oracle on a bounded sample per step"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cases", action="store_true", help="headline step only")
    ap.add_argument("--gemm-m", type=int, default=0, help="gemm workload: only this M")
    ap.add_argument("--cpu-budget-s", type=float, default=3.0,
                    help="reference arm: seconds of oracle attention work sampled per step")
    ap.add_argument("--workload", default="step",
                    choices=["step", "all", *CASE_GROUPS, "attention-small", "attention-small-d15",
                             "attention-largeg-small", "logits-small", "adasd-small", "accept-one"],
                    help="step: the headline line (with all cases); others print one JSON line per case")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1 or args.gpus != 1:
        # one GPU per process and no multi-GPU path: nothing is launched
        if rank == 0:
            print(json.dumps({"impl": "ours", "metric": METRIC, "n_gpus": max(world, args.gpus),
                              "unavailable": "the verification path is built for one GPU; "
                                             "there is no multi-GPU arm"}), flush=True)
        return
    if args.workload != "step":
        case_lines(args)
        return
    line = gpu_arm(args)
    if not args.no_cpu_baseline:
        t, s, desc, nthreads = cpu_sample_time()
        v = WORKLOAD["B"] * (1 + WORKLOAD["D"]) / t
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                                "sample": desc, "sampled_s": s, "value_kind": "extrapolated from the sample"}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
