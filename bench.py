#!/usr/bin/env python
"""Benchmark of the quantized self-speculative hot path on GB300.

A step is one speculative round over the LLaMA-2-7B-shaped linears
(32 layers x {q, k, v, o 4096x4096; gate, up 4096->11008; down 11008->4096}
+ lm_head 4096->32000), nested 4+4-bit weights, group 128, batch 1, k = 4:
  4 draft passes   : every linear, base plane only, M = 1 (one persistent launch each)
  1 verify pass    : every linear, both planes (8-bit target), M = k+1 = 5
  acceptance       : greedy and sampled (T = 1) on the lm_head outputs, V = 32000
Value = algorithmic HBM bytes of the round / device time (GB/s), whole job.
Synthetic, seeded inputs; the packed weights (6.8 GB) exceed L2, so every
pass streams from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "nested-quant draft GEMV / verify GEMM HBM GB/s (% of peak); accept rounds/s"
WORKLOAD = "llama2-7b-linears-32L-g128-b1-k4"
K_DRAFT = 4
GROUP = 128
V_LM = 32000


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


NOMINAL_HBM_GBS = 8000.0   # HBM3e nominal, reported beside the measured-peak fraction


def bf16_peak_tflops():
    """Measured dense bf16 (= fp16) tensor throughput, burst; fallback 1900."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (read-only queries)."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) != len(self.FIELDS):
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[3:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ model
def linear_list():
    from quantized_self_speculative_gb300 import synth
    layer, lm, n_layers = synth.llama2_7b_linears()
    shapes = []
    for li in range(n_layers):
        for name, n, k in layer:
            shapes.append((f"L{li}.{name}", n, k))
    shapes.append((lm[0], lm[1], lm[2]))
    return shapes


def draft_bytes(n, k, M, g=GROUP):
    return n * k // 2 + 2 * n * k // g + M * k * 2 + M * n * 4


def verify_bytes(n, k, M, g=GROUP):
    return n * k + 2 * n * k // g + M * k * 2 + M * n * 4


def accept_bytes(B, k, V, sampled):
    return B * ((2 * k + 1) if sampled else (k + 1)) * V * 4 + B * k * 4 + B * (k + 2) * 4


class Round:
    """Device state of one speculative round (weights resident in HBM)."""

    def __init__(self, device, seed=0):
        import torch
        from quantized_self_speculative_gb300 import nq
        self.torch, self.nq = torch, nq
        self.dev = device
        self.shapes = linear_list()
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        self.layers = []
        for _, n, k in self.shapes:
            w = torch.randn((n, k), generator=gen, device=device, dtype=torch.float32).mul_(0.02)
            self.layers.append(nq.pack_weights(w, nq.FMT_NESTED44, GROUP))
            del w
        torch.cuda.synchronize()
        # activations: one slab per round (q/k/v share an input, gate/up share one)
        M_v = K_DRAFT + 1
        specs = []   # (pass, layer index, M, k)
        for p in range(K_DRAFT):
            specs += [(p, i, 1, k) for i, (_, n, k) in enumerate(self.shapes)]
        specs += [(K_DRAFT, i, M_v, k) for i, (_, n, k) in enumerate(self.shapes)]
        offsets, total, cache = {}, 0, {}
        for p, i, M, k in specs:
            name = self.shapes[i][0]
            key = (p, name.split(".")[0], "qkv" if name.endswith((".q", ".k", ".v")) else
                   "gu" if name.endswith((".gate", ".up")) else name)
            if key not in cache:
                cache[key] = total
                total += M * k
            offsets[(p, i)] = cache[key]
        self.x_host = torch.empty(total, dtype=torch.bfloat16).pin_memory()
        self.x_host.copy_(torch.randn(total, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16))
        self.x_dev = self.x_host.to(device)
        self.h2d_bytes = total * 2
        self.dl = torch.empty((1, K_DRAFT, V_LM), dtype=torch.float32, device=device)
        self.tl = torch.empty((1, K_DRAFT + 1, V_LM), dtype=torch.float32, device=device)
        self.batches = []
        for p in range(K_DRAFT + 1):
            M = 1 if p < K_DRAFT else M_v
            xs, ys = [], []
            for i, (name, n, k) in enumerate(self.shapes):
                o = offsets[(p, i)]
                xs.append(self.x_dev[o:o + M * k].view(M, k))
                if name == "lm_head":
                    ys.append(self.dl[0, p:p + 1] if p < K_DRAFT else self.tl[0])
                else:
                    ys.append(torch.empty((M, n), dtype=torch.float32, device=device))
            self.batches.append(nq.LinearBatch(p == K_DRAFT, self.layers, xs, ys))
        # target-only decoding step for Eq. (2)'s baseline: the 8-bit target (both
        # planes) over one token per pass (M = 1), same weights and activations
        self.target_only = nq.LinearBatch(True, self.layers, self.batches[0]._keep[1],
                                          [torch.empty((1, n), dtype=torch.float32, device=device)
                                           for _, n, _ in self.shapes])
        g = np.random.default_rng(seed + 2)
        self.draft = torch.from_numpy(g.integers(0, V_LM, size=(1, K_DRAFT), dtype=np.int32)).to(device)
        self.seeds = torch.from_numpy(np.array([seed + 3], dtype=np.int64)).to(device)
        self.ws_g = nq.accept_workspace(1, K_DRAFT, V_LM, device)
        self.ws_s = nq.accept_workspace(1, K_DRAFT, V_LM, device)
        self.out_g = torch.empty((1, K_DRAFT + 1), dtype=torch.int32, device=device)
        self.cnt_g = torch.empty(1, dtype=torch.int32, device=device)
        self.out_s = torch.empty((1, K_DRAFT + 1), dtype=torch.int32, device=device)
        self.cnt_s = torch.empty(1, dtype=torch.int32, device=device)
        self.res_host = torch.empty(2 * (K_DRAFT + 2), dtype=torch.int32).pin_memory()
        self.round_idx = 0
        self.bytes_draft_pass = sum(draft_bytes(n, k, 1) for _, n, k in self.shapes)
        self.bytes_verify = sum(verify_bytes(n, k, M_v) for _, n, k in self.shapes)
        self.bytes_accept = accept_bytes(1, K_DRAFT, V_LM, False) + accept_bytes(1, K_DRAFT, V_LM, True)
        self.bytes_round = K_DRAFT * self.bytes_draft_pass + self.bytes_verify + self.bytes_accept
        # k draft passes + 1 verify pass + greedy (1 kernel) + sampled acceptance
        # (3 kernels: segment pass, decisions, resample pass)
        self.launches_per_round = K_DRAFT + 1 + 1 + 3

    def run(self, events=None):
        nq = self.nq
        for p in range(K_DRAFT + 1):
            if events is not None:
                events[p].record()
            self.batches[p]()
        if events is not None:
            events[K_DRAFT + 1].record()
        nq.accept_greedy(self.draft, self.tl, ws=self.ws_g, out_tok=self.out_g, out_cnt=self.cnt_g)
        nq.accept_sample(self.draft, self.dl, self.tl, 1.0, self.seeds, self.round_idx, ws=self.ws_s,
                         out_tok=self.out_s, out_cnt=self.cnt_s)
        if events is not None:
            events[K_DRAFT + 2].record()
        self.round_idx += 1

    def run_e2e(self):
        """The same round through the public API with host buffers: the round's
        activations come from pinned host memory; the emitted tokens return."""
        torch = self.torch
        self.x_dev.copy_(self.x_host, non_blocking=True)
        self.run()
        self.res_host[0:K_DRAFT + 1].copy_(self.out_g[0], non_blocking=True)
        self.res_host[K_DRAFT + 1:K_DRAFT + 2].copy_(self.cnt_g, non_blocking=True)
        self.res_host[K_DRAFT + 2:2 * K_DRAFT + 3].copy_(self.out_s[0], non_blocking=True)
        self.res_host[2 * K_DRAFT + 3:2 * K_DRAFT + 4].copy_(self.cnt_s, non_blocking=True)
        return self.res_host

    @property
    def d2h_bytes(self):
        return 2 * (K_DRAFT + 2) * 4

    def time_target_only(self, iters=20):
        torch = self.torch
        for _ in range(3):
            self.target_only()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            self.target_only()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / iters


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one draft-pass
# launch of the streaming kernel at this workload: an ncu capture of the
# 8-layer case (0.999x its algorithmic bytes) scaled to the 32 layers + lm_head
# by the algorithmic 3,414,627,328 B (no re-reads).  Set to None whenever that
# kernel changes until it is captured again.
DRAFT_PASS_DRAM_BYTES = 3_412_049_000


def eq2_report(t_draft_us, t_verify_us, t_accept_us, t_target_us, k=K_DRAFT):
    """Erge, "Tokens per pass and time per token": Eq. (1) gives the expected
    tokens per target pass E = (1 - a^(k+1)) / (1 - a) at acceptance rate a,
    Eq. (2) the time per token t = (t_pass + k t_draft) / E, from the measured
    pass times (t_pass = verify pass + acceptance).  The baseline is the
    target alone, one token per pass (verify linears at M = 1)."""
    t_pass = t_verify_us + t_accept_us
    out = {"k": k, "t_draft_us": round(t_draft_us, 1), "t_pass_us": round(t_pass, 1),
           "t_target_only_us": round(t_target_us, 1), "by_alpha": {}}
    for a in (0.46, 0.6, 0.88, 0.95):
        E = (1 - a ** (k + 1)) / (1 - a)
        t = (t_pass + k * t_draft_us) / E
        out["by_alpha"][str(a)] = {"tokens_per_pass": round(E, 3), "t_token_us": round(t, 1),
                                   "speedup_vs_target_only": round(t_target_us / t, 3)}
    return out


# ------------------------------------------------------------------ the round, measured
class RoundLoop:
    """Whole speculative rounds on the device ("Drafting and checking
    tokens"; Eq. (2)): LLaMA-2-7B-shaped linears with q|k|v and gate|up fused
    (one weight stream per layer input: 32 x {qkv 4096->12288, o 4096x4096,
    gate|up 4096->22016, down 11008->4096} + lm_head 4096->32000), nested
    4+4-bit, group 128, batch 1, k = 4, greedy.  Per round: k draft passes
    (base plane, M = 1), each drafted token the argmax of the previous draft
    pass's lm_head output and the next pass's lm_head input (its embedding
    row); one verify pass over the k+1 positions (both planes, M = k+1); greedy
    acceptance; the emitted tokens committed on the device.  The linears other
    than lm_head take fixed synthetic activations (the attention, norms and
    MLP nonlinearity between linears are not part of this hot path), so the
    token dependency runs through lm_head.  One round is captured in a CUDA
    graph and replayed; the emitted count is read back once at the end."""

    def __init__(self, device, seed=23, k=K_DRAFT, max_rounds=512):
        import torch
        from quantized_self_speculative_gb300 import nq
        self.torch, self.nq, self.dev, self.k = torch, nq, device, k
        h, f = 4096, 11008
        layer = [("qkv", 3 * h, h), ("o", h, h), ("gate_up", 2 * f, h), ("down", h, f)]
        self.shapes = [(f"L{i}.{nm}", n, kk) for i in range(32) for nm, n, kk in layer] + [("lm_head", V_LM, h)]
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        self.layers = []
        for _, n, kk in self.shapes:
            w = torch.randn((n, kk), generator=gen, device=device, dtype=torch.float32).mul_(0.02)
            self.layers.append(nq.pack_weights(w, nq.FMT_NESTED44, GROUP))
            del w
        self.table = torch.randn((V_LM, h), generator=gen, device=device).to(torch.bfloat16)
        B = 1
        self.x_lm = torch.empty((B, h), dtype=torch.bfloat16, device=device)
        self.y_lm = torch.empty((B, V_LM), dtype=torch.float32, device=device)
        self.x_v = torch.empty((B * (k + 1), h), dtype=torch.bfloat16, device=device)
        self.tl = torch.empty((B, k + 1, V_LM), dtype=torch.float32, device=device)

        def batch(M, x_last, y_last, verify):
            xs, ys = [], []
            for name, n, kk in self.shapes:
                if name == "lm_head":
                    xs.append(x_last)
                    ys.append(y_last)
                else:
                    xs.append(torch.randn((M, kk), generator=gen, device=device).to(torch.bfloat16))
                    ys.append(torch.empty((M, n), dtype=torch.float32, device=device))
            return nq.LinearBatch(verify, self.layers, xs, ys)
        self.draft_batch = batch(B, self.x_lm, self.y_lm, False)
        self.verify_batch = batch(B * (k + 1), self.x_v, self.tl.view(B * (k + 1), V_LM), True)
        self.target_batch = batch(B, self.x_lm, self.y_lm, True)
        self.max_len = 1 + max_rounds * (k + 1)
        self.seq = torch.full((B, self.max_len), -1, dtype=torch.int32, device=device)
        self.seq_len = torch.ones(B, dtype=torch.int32, device=device)
        self.x0 = torch.tensor([7], dtype=torch.int32, device=device)
        self.seq[0, 0] = 7
        self.draft = torch.zeros((B, k), dtype=torch.int32, device=device)
        self.out_tok = torch.empty((B, k + 1), dtype=torch.int32, device=device)
        self.out_cnt = torch.empty(B, dtype=torch.int32, device=device)
        self.ws_arg = nq.accept_workspace(B, 0, V_LM, device)
        self.ws_acc = nq.accept_workspace(B, k, V_LM, device)
        self.bytes_draft = sum(draft_bytes(n, kk, 1) for _, n, kk in self.shapes)
        self.bytes_verify = sum(verify_bytes(n, kk, k + 1) for _, n, kk in self.shapes)
        self.graph = None

    def one_round(self, ev=None):
        nq, k = self.nq, self.k
        for j in range(k):
            if ev is not None:
                ev[j].record()
            if j == 0:
                nq.embed_rows(self.table, self.x0, 1, out=self.x_lm)
            else:
                nq.embed_rows(self.table, self.draft.view(-1)[j - 1:], 1, ids_stride=k, out=self.x_lm)
            self.draft_batch()
            nq.draft_argmax(self.y_lm, self.draft.view(-1)[j:], tok_stride=k, ws=self.ws_arg)
        if ev is not None:
            ev[k].record()
        nq.embed_round(self.table, self.x0, self.draft, 1, k, out=self.x_v)
        self.verify_batch()
        if ev is not None:
            ev[k + 1].record()
        nq.accept_greedy(self.draft, self.tl, ws=self.ws_acc, out_tok=self.out_tok, out_cnt=self.out_cnt)
        nq.round_commit(self.out_tok, self.out_cnt, self.seq, self.seq_len, self.x0)
        if ev is not None:
            ev[k + 2].record()

    def reset(self):
        self.seq_len.fill_(1)
        self.x0.fill_(7)

    def capture(self):
        torch = self.torch
        self.one_round()                      # warm-up outside the capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=s):
                self.one_round()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def measure(self, rounds=100):
        """Rounds replayed from the graph; time per round and per emitted token,
        with the pass times of the same round (events, eager) for Eq. (2)."""
        torch, k = self.torch, self.k
        if self.graph is None:
            self.capture()
        self.reset()
        for _ in range(3):
            self.graph.replay()
        self.reset()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(rounds):
            self.graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us_round = e0.elapsed_time(e1) * 1e3 / rounds
        tokens = int(self.seq_len[0].item()) - 1
        # pass times of the same round (eager, events between the launches)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(k + 3)] for _ in range(10)]
        for ev in evs:
            self.one_round(ev)
        torch.cuda.synchronize()
        t_draft = statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in evs for j in range(k)) * 1e3
        t_verify = statistics.mean(ev[k].elapsed_time(ev[k + 1]) for ev in evs) * 1e3
        t_accept = statistics.mean(ev[k + 1].elapsed_time(ev[k + 2]) for ev in evs) * 1e3
        # the target alone: one verify pass over one position per token (M = 1)
        for _ in range(3):
            self.target_batch()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(20):
            self.target_batch()
        e1.record()
        torch.cuda.synchronize()
        t_target = e0.elapsed_time(e1) * 1e3 / 20
        E = tokens / rounds
        # acceptance rate implied by Eq. (1) at the measured tokens per round
        lo, hi = 0.0, 1.0
        for _ in range(60):
            a = 0.5 * (lo + hi)
            if (1 - a ** (k + 1)) / (1 - a) < E:
                lo = a
            else:
                hi = a
        alpha = 0.5 * (lo + hi)
        eq2 = (t_verify + t_accept + k * t_draft) / E
        return {"rounds": rounds, "tokens": tokens, "tokens_per_round": round(E, 4),
                "alpha_from_eq1": round(alpha, 4), "us_per_round": round(us_round, 1),
                "us_per_token": round(us_round / E, 1),
                "eq2_us_per_token_from_pass_times": round(eq2, 1),
                "t_draft_pass_us": round(t_draft, 1), "t_verify_pass_us": round(t_verify, 1),
                "t_accept_commit_us": round(t_accept, 1), "t_target_only_us": round(t_target, 1),
                "speedup_vs_target_only": round(t_target / (us_round / E), 3),
                "draft_pass_gbs": round(self.bytes_draft / (t_draft * 1e-6) / 1e9, 1),
                "verify_pass_gbs": round(self.bytes_verify / (t_verify * 1e-6) / 1e9, 1),
                "layout": "q|k|v and gate|up fused: 129 linears per pass",
                "launches_per_round": 3 * k + 5}


# ------------------------------------------------------------------ int8 activations (W4A8 -> W8A8)
def a8_sweep(device, iters=10):
    """BitNest's own precision (Table 1, "W4A8 -> W8A8"): the LLaMA-2-7B pass
    with int8 activation codes, draft at M = 1 (base plane) and verify at
    M = k+1 = 5 (both planes), exact group dots on the streaming weight kernel
    (warp MMA); plus the per-row activation quantiser over one [M][4096] input
    (100 back-to-back calls, launch overhead included).  Algorithmic bytes
    as for the bf16-activation passes with 1-byte activations."""
    import torch
    from quantized_self_speculative_gb300 import nq, synth
    hbm, _ = peaks()
    shapes = _shapes(synth.llama2_7b_linears)
    layers = _pass_layers(device, shapes, nq.FMT_NESTED44, GROUP, 97)
    out = {}
    gen = torch.Generator(device=device)
    gen.manual_seed(98)
    for kind, M, verify in (("draft_w4a8_M1", 1, False), ("verify_w8a8_M5", K_DRAFT + 1, True)):
        xqs, sxs, ys = [], [], []
        for L in layers:
            x = torch.randn((M, L.k_in), generator=gen, device=device).to(torch.bfloat16)
            xq, sx = nq.quantize_act_int8(x)
            xqs.append(xq)
            sxs.append(sx)
            ys.append(torch.empty((M, L.n_out), dtype=torch.float32, device=device))
        b = nq.LinearA8Batch(verify, layers, xqs, sxs, ys)
        for _ in range(3):
            b()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            b()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / iters
        w = 1.0 if verify else 0.5
        byts = sum(w * L.n_out * L.k_in + 2 * L.n_out * L.k_in // GROUP + M * L.k_in + 4 * M + 4 * M * L.n_out
                   for L in layers)
        out[kind] = {"us": round(us, 1), "gbs": round(byts / (us * 1e-6) / 1e9, 1),
                     "frac": round(byts / (us * 1e-6) / 1e9 / hbm, 4), "bytes": int(byts)}
        x = torch.randn((M, 4096), generator=gen, device=device).to(torch.bfloat16)
        xq = torch.empty((M, 4096), dtype=torch.int8, device=device)
        sx = torch.empty(M, dtype=torch.float32, device=device)
        e0.record()
        for _ in range(100):
            nq.quantize_act_int8(x, xq, sx)
        e1.record()
        torch.cuda.synchronize()
        out[kind]["quantize_act_us_per_input"] = round(e0.elapsed_time(e1) * 1e3 / 100, 2)
    del layers
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ nested KV cache attention (long context)
def kv_sweep(device, ctx=32768, layers=4, iters=10):
    """Decode attention over the nested KV cache at a 32K context, batch 1
    (BitNest Fig. 4-5, Tables 9-10: the draft reads the KV4 base view, the
    verify pass the KV8 view): LLaMA-2-7B-32K heads (32 x 128, MHA) and
    Qwen2.5-7B heads (28 query / 4 kv heads x 128, GQA).  Four layers' caches
    are rotated so that every call streams from HBM.  Algorithmic bytes per
    call: K and V rows read, len x (planes x d/2 + 2 d/G) each, plus q and out."""
    import torch
    from quantized_self_speculative_gb300 import nq
    hbm, _ = peaks()
    out = {}
    gen = torch.Generator(device=device)
    gen.manual_seed(71)
    for name, Hq, Hkv in (("llama2_7b_32k_mha", 32, 32), ("qwen25_7b_gqa", 28, 4)):
        d, G = 128, 128
        caches = [nq.KVCache(1, Hkv, d, G, ctx + 16, device) for _ in range(layers)]
        for c in caches:
            for lo in range(0, ctx, 4096):
                k = torch.randn((1, Hkv, 4096, d), generator=gen, device=device)
                v = torch.randn((1, Hkv, 4096, d), generator=gen, device=device)
                c.append(k, v, torch.tensor([lo], dtype=torch.int32, device=device))
        torch.cuda.synchronize()
        res = {}
        for kind, M, planes in (("draft_M1_kv4", 1, 1), ("verify_M5_kv8", K_DRAFT + 1, 2)):
            q = torch.randn((1, M, Hq, d), generator=gen, device=device)
            lens = torch.tensor([ctx], dtype=torch.int32, device=device)
            o = torch.empty_like(q)
            need = nq.lib().nq_attn_workspace_bytes(1, M, Hq, d, ctx + 16)
            ws = torch.empty(need, dtype=torch.uint8, device=device)
            for c in caches:
                c.attention(q, lens, planes, d ** -0.5, out=o, ws=ws)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(iters):
                for c in caches:
                    c.attention(q, lens, planes, d ** -0.5, out=o, ws=ws)
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (iters * layers)
            byts = 2 * Hkv * ctx * (planes * d // 2 + 2 * d // G) + 2 * M * Hq * d * 4
            res[kind] = {"us_per_layer": round(us, 2), "gbs": round(byts / (us * 1e-6) / 1e9, 1),
                         "frac": round(byts / (us * 1e-6) / 1e9 / hbm, 4), "bytes": byts}
        res["draft_speedup_kv4_vs_kv8_per_row"] = round(res["verify_M5_kv8"]["us_per_layer"] /
                                                       res["draft_M1_kv4"]["us_per_layer"], 3)
        out[name] = res
        del caches
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ per-linear times (LLaMA-2-7B shapes)
def per_linear_table(R, reps=3):
    """Device time of one linear per launch, for each linear shape of the
    round: the 32 layer copies of the shape (their weights exceed L2 together)
    run back to back as single-linear calls inside a CUDA graph; time per
    launch = graph time / 32.  Draft (M = 1, base plane) and verify (M = 5,
    both planes).  The whole-pass figures come from one persistent launch over
    all 225 linears, which hides the per-launch gaps these numbers include."""
    import torch
    nq = R.nq
    groups = {"q/k/v/o 4096x4096": (".q", ".k", ".v", ".o"), "gate/up 4096->11008": (".gate", ".up"),
              "down 11008->4096": (".down",), "lm_head 4096->32000": ("lm_head",)}
    out = {}
    for name, suffixes in groups.items():
        idx = [i for i, (nm, _, _) in enumerate(R.shapes) if nm.endswith(suffixes)][:32]
        n, k = R.shapes[idx[0]][1], R.shapes[idx[0]][2]
        row = {"n_out": n, "k_in": k, "launches": len(idx)}
        for kind, M in (("draft_M1", 1), ("verify_M5", 5)):
            verify = kind.startswith("verify")
            x = torch.randn((M, k), device=R.dev).to(torch.bfloat16)
            y = torch.empty((M, n), dtype=torch.float32, device=R.dev)
            fn = nq.verify_gemm if verify else nq.draft_gemv
            for i in idx:                                   # warm-up outside capture
                fn(R.layers[i], x, y)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in idx:
                    fn(R.layers[i], x, y)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps * len(idx))
            byts = (verify_bytes if verify else draft_bytes)(n, k, M)
            row[kind] = {"us": round(us, 2), "gbs": round(byts / (us * 1e-6) / 1e9, 1), "bytes": byts}
        out[name] = row
    return out


# ------------------------------------------------------------------ acceptance at the sweep shape
def accept_sweep(device, iters=20, ks=(2, 4, 6, 8)):
    """Acceptance kernels alone at B = 64, V = 152064 (fp32 logits ~ N(0, 3),
    draft = target + N(0, 0.3)), k in {2, 4, 6, 8}."""
    import torch
    from quantized_self_speculative_gb300 import nq
    out = {}
    B, V = 64, 152064
    gen = torch.Generator(device=device)
    gen.manual_seed(5)
    for k in ks:
        tl = torch.randn((B, k + 1, V), generator=gen, device=device).mul_(3.0)
        dl = (tl[:, :k] + 0.3 * torch.randn((B, k, V), generator=gen, device=device)).contiguous()
        d = dl.argmax(-1).to(torch.int32)
        seeds = torch.arange(B, dtype=torch.int64, device=device)
        ws = nq.accept_workspace(B, k, V, device)
        res = {}
        for kind in ("greedy", "sample"):
            def call(r):
                if kind == "greedy":
                    nq.accept_greedy(d, tl, ws=ws)
                else:
                    nq.accept_sample(d, dl, tl, 1.0, seeds, r, ws=ws)
            for r in range(3):
                call(r)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for r in range(iters):
                call(r)
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / iters
            byts = accept_bytes(B, k, V, kind == "sample")
            gbs = byts / (us * 1e-6) / 1e9
            res[kind] = {"us": round(us, 2), "rounds_per_s": round(B / (us * 1e-6), 1),
                         "gbs": round(gbs, 1), "frac": round(gbs / peaks()[0], 4)}
        out[f"k{k}"] = res
        del tl, dl
    return out


# ------------------------------------------------------------------ whole-pass sweeps (configs 3 and 4)
def _pass_layers(device, shapes, fmt, group, seed, w16=False):
    """Pack every linear of a pass in one format (weights drawn on the GPU)."""
    import torch
    from quantized_self_speculative_gb300 import nq
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    layers = []
    for n, k in shapes:
        w = torch.randn((n, k), generator=gen, device=device, dtype=torch.float32).mul_(0.02)
        if w16:
            w = w.half().float()          # the tiers derive from one fp16 base
        layers.append(nq.pack_weights(w, fmt, group))
        del w
    torch.cuda.synchronize()
    return layers


def _time_pass(device, layers, M, verify, iters=10, tensor_cores=False):
    """Device time of one batched call over all layers at M activation rows
    (tensor_cores: the *_ws entry point, tensor-memory kernel at M >= 16,
    including its activation pre-pass)."""
    import torch
    from quantized_self_speculative_gb300 import nq
    gen = torch.Generator(device=device)
    gen.manual_seed(123)
    xs = [torch.randn((M, L.k_in), generator=gen, device=device).to(torch.bfloat16) for L in layers]
    ys = [torch.empty((M, L.n_out), dtype=torch.float32, device=device) for L in layers]
    b = nq.LinearBatch(verify, layers, xs, ys, tensor_cores=tensor_cores)
    for _ in range(3):
        b()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        b()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / iters
    per_w = {nq.FMT_NESTED44: (1.0 if verify else 0.5), nq.FMT_INT4: 0.5, nq.FMT_FP8E4M3_ROW: 1.0, nq.FMT_FP16: 2.0}
    byts = 0
    for L in layers:
        wb = per_w[L.fmt] * L.n_out * L.k_in
        sb = (2 * L.n_out * L.k_in // L.group) if L.fmt in (nq.FMT_NESTED44, nq.FMT_INT4) else (4 * L.n_out if L.fmt == nq.FMT_FP8E4M3_ROW else 0)
        byts += wb + sb + 2 * M * L.k_in + 4 * M * L.n_out
    hbm, _ = peaks()
    tflops = 2.0 * M * sum(L.n_out * L.k_in for L in layers) / (us * 1e-6) / 1e12
    return {"M": M, "us": round(us, 1), "gbs": round(byts / (us * 1e-6) / 1e9, 1),
            "frac": round(byts / (us * 1e-6) / 1e9 / hbm, 4),
            "frac_nominal": round(byts / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4), "bytes": int(byts),
            "tflops": round(tflops, 2), "frac_tensor": round(tflops / bf16_peak_tflops(), 4)}


def _shapes(spec):
    layer, lm, n_layers = spec()
    return [(n, k) for _ in range(n_layers) for _, n, k in layer] + [(lm[1], lm[2])]


def config3_sweep(device):
    """LLaMA-3-8B-shaped linears, batch 16, k = 8: draft M = 16 (base plane),
    verify M = 144 (both planes), groups 64 and 128; the tensor-memory kernel
    (the *_ws entry points) and, for comparison, the streaming kernel."""
    import torch
    from quantized_self_speculative_gb300 import nq, synth
    out = {}
    shapes = _shapes(synth.llama3_8b_linears)
    for g in (128, 64):
        layers = _pass_layers(device, shapes, nq.FMT_NESTED44, g, 31 + g)
        out[f"g{g}"] = {"draft_M16": _time_pass(device, layers, 16, False, tensor_cores=True),
                        "verify_M144": _time_pass(device, layers, 144, True, tensor_cores=True),
                        "draft_M16_stream_kernel": _time_pass(device, layers, 16, False),
                        "verify_M144_stream_kernel": _time_pass(device, layers, 144, True, iters=2)}
        del layers
        torch.cuda.empty_cache()
    return out


def config4_sweep(device):
    """Qwen2.5-7B-shaped linears (28 layers), three tiers of one fp16 base:
    INT4 g128 draft at M = 1; FP8 (row scale) and FP16 verify at M = k+1."""
    import torch
    from quantized_self_speculative_gb300 import nq, synth
    shapes = _shapes(synth.qwen25_7b_linears)
    out = {}
    int4 = _pass_layers(device, shapes, nq.FMT_INT4, 128, 41, w16=True)
    out["int4_draft_M1"] = _time_pass(device, int4, 1, False)
    del int4
    for name, fmt in (("fp8_verify", nq.FMT_FP8E4M3_ROW), ("fp16_verify", nq.FMT_FP16)):
        layers = _pass_layers(device, shapes, fmt, 0, 41, w16=True)
        out[name] = {f"k{k}": _time_pass(device, layers, k + 1, True) for k in (2, 4, 6, 8)}
        del layers
        torch.cuda.empty_cache()
    return out


def _alpha_hat(device, gen, B, k, V, sigma, rounds, seed_base, nq, ws):
    """Measured acceptance rate (accepted / tested positions) of sampled
    acceptance, target logits ~ N(0, 3), draft = target + N(0, sigma), T = 1."""
    import torch
    seeds = torch.arange(B, dtype=torch.int64, device=device) + seed_base
    acc_pos, tested, tot = 0, 0, 0
    for r in range(rounds):
        tl = torch.randn((B, k + 1, V), generator=gen, device=device).mul_(3.0)
        dl = (tl[:, :k] + sigma * torch.randn((B, k, V), generator=gen, device=device)).contiguous()
        p = torch.softmax(dl.double(), -1).view(-1, V)
        d = torch.multinomial(p, 1, generator=gen).view(B, k).to(torch.int32)
        _, cnt = nq.accept_sample(d, dl, tl, 1.0, seeds, r, ws=ws)
        c = cnt.to(torch.int64)
        tot += int(c.sum())
        acc_pos += int((c - 1).sum())
        tested += int(torch.minimum(c, torch.full_like(c, k)).sum())
    return acc_pos / max(1, tested), tot


def config5_tokens(device, rounds=200):
    """Acceptance sweep semantics: draft noise sigma calibrated (bisection on a
    short pilot) to acceptance rates of about 0.6 and 0.95; then mean tokens
    per sampled round vs Eq. (1) at the measured rate, and greedy rounds,
    B = 64, V = 152064, T = 1, k in {2, 4, 6, 8}."""
    import math
    import torch
    from quantized_self_speculative_gb300 import nq
    B, V = 64, 152064
    gen = torch.Generator(device=device)
    out = {}
    ws4 = nq.accept_workspace(B, 4, V, device)
    for target in (0.6, 0.95):
        lo, hi = math.log(0.01), math.log(8.0)   # alpha falls as sigma grows
        for it in range(9):
            mid = 0.5 * (lo + hi)
            gen.manual_seed(77 + it)
            a, _ = _alpha_hat(device, gen, B, 4, V, math.exp(mid), 20, 500, nq, ws4)
            if a > target:
                lo = mid
            else:
                hi = mid
        sigma = math.exp(0.5 * (lo + hi))
        for k in (2, 4, 6, 8):
            gen.manual_seed(1000 * k + int(target * 100))
            ws = nq.accept_workspace(B, k, V, device)
            seeds = torch.arange(B, dtype=torch.int64, device=device) + 1000 * k
            tot_s, acc_pos, tested, tot_g = 0, 0, 0, 0
            for r in range(rounds):
                tl = torch.randn((B, k + 1, V), generator=gen, device=device).mul_(3.0)
                dl = (tl[:, :k] + sigma * torch.randn((B, k, V), generator=gen, device=device)).contiguous()
                p = torch.softmax(dl.double(), -1).view(-1, V)
                d = torch.multinomial(p, 1, generator=gen).view(B, k).to(torch.int32)
                _, cnt = nq.accept_sample(d, dl, tl, 1.0, seeds, r, ws=ws)
                _, cntg = nq.accept_greedy(dl.argmax(-1).to(torch.int32), tl, ws=ws)
                c = cnt.to(torch.int64)
                tot_s += int(c.sum())
                tot_g += int(cntg.sum())
                acc_pos += int((c - 1).sum())
                tested += int(torch.minimum(c, torch.full_like(c, k)).sum())
            alpha = acc_pos / max(1, tested)
            e1 = (1 - alpha ** (k + 1)) / (1 - alpha) if alpha < 1 else k + 1
            out[f"alpha{target}_k{k}"] = {"sigma": round(sigma, 4), "alpha_hat": round(alpha, 4),
                                          "tokens_per_round_sampled": round(tot_s / (rounds * B), 4),
                                          "eq1_at_alpha_hat": round(e1, 4),
                                          "tokens_per_round_greedy": round(tot_g / (rounds * B), 4),
                                          "rounds": rounds * B}
    return out


def profile_case(case, layers=8):
    """Small fixed workloads for ncu captures: a few launches of one kernel."""
    import torch
    from quantized_self_speculative_gb300 import build, nq, synth
    build.build()
    device = torch.device("cuda")
    if case in ("draft", "verify", "draft16", "verify144", "int4", "fp8", "fp16"):
        spec = synth.llama3_8b_linears if case in ("draft16", "verify144") else (
            synth.qwen25_7b_linears if case in ("int4", "fp8", "fp16") else synth.llama2_7b_linears)
        layer, _, _ = spec()
        shapes = [(n, k) for _ in range(layers) for _, n, k in layer]
        fmt = {"int4": nq.FMT_INT4, "fp8": nq.FMT_FP8E4M3_ROW, "fp16": nq.FMT_FP16}.get(case, nq.FMT_NESTED44)
        L = _pass_layers(device, shapes, fmt, 128 if fmt in (nq.FMT_NESTED44, nq.FMT_INT4) else 0, 1)
        M = {"draft": 1, "verify": 5, "draft16": 16, "verify144": 144, "int4": 1, "fp8": 5, "fp16": 5}[case]
        print(json.dumps({"case": case, **_time_pass(device, L, M, case not in ("draft", "draft16", "int4"), iters=2,
                                                      tensor_cores=case in ("draft16", "verify144"))}))
    elif case in ("kv4", "kv8"):
        # one LLaMA-2-7B-32K layer's cache (32 kv heads x 128, 32K rows; 276 MB
        # of planes, beyond L2), the draft (KV4, M = 1) or verify (KV8, M = 5) read
        planes = 1 if case == "kv4" else 2
        M, ctx, H, d = (1 if planes == 1 else K_DRAFT + 1), 32768, 32, 128
        gen = torch.Generator(device=device)
        gen.manual_seed(5)
        c = nq.KVCache(1, H, d, GROUP, ctx + 16, device)
        for lo in range(0, ctx, 4096):
            kv = torch.randn((1, H, 4096, d), generator=gen, device=device)
            c.append(kv, kv, torch.tensor([lo], dtype=torch.int32, device=device))
        q = torch.randn((1, M, H, d), generator=gen, device=device)
        lens = torch.tensor([ctx], dtype=torch.int32, device=device)
        out = torch.empty_like(q)
        ws = torch.empty(nq.lib().nq_attn_workspace_bytes(1, M, H, d, ctx + 16), dtype=torch.uint8, device=device)
        for _ in range(3):
            c.attention(q, lens, planes, d ** -0.5, out=out, ws=ws)
        torch.cuda.synchronize()
        print(json.dumps({"case": case, "ctx": ctx, "heads": H, "M": M}))
    else:
        B, k, V = 64, 4, 152064
        gen = torch.Generator(device=device)
        gen.manual_seed(1)
        tl = torch.randn((B, k + 1, V), generator=gen, device=device).mul_(3.0)
        dl = (tl[:, :k] + 0.3 * torch.randn((B, k, V), generator=gen, device=device)).contiguous()
        d = dl.argmax(-1).to(torch.int32)
        seeds = torch.arange(B, dtype=torch.int64, device=device)
        ws = nq.accept_workspace(B, k, V)
        for r in range(4):
            if case == "greedy":
                nq.accept_greedy(d, tl, ws=ws)
            else:
                nq.accept_sample(d, dl, tl, 1.0, seeds, r, ws=ws)
        torch.cuda.synchronize()
        print(json.dumps({"case": case, "B": B, "k": k, "V": V}))


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample_step(state):
    """A bounded sample of the round on the CPU oracle: draft (M=1) and verify
    (M=5) of the q, gate and down linears, plus greedy and sampled acceptance
    at V = 32000.  Returns algorithmic bytes processed."""
    import oracle as O
    from quantized_self_speculative_gb300 import synth
    if "packed" not in state:
        packed = []
        for i, (n, k) in enumerate([(4096, 4096), (11008, 4096), (4096, 11008)]):
            w = synth.weights(9000 + i, n, k)
            packed.append((n, k) + O.pack_nested(w, GROUP))
        state["packed"] = packed
        state["x1"] = {k: synth.activations_bf16(9100 + k, 1, k) for k in (4096, 11008)}
        state["x5"] = {k: synth.activations_bf16(9200 + k, 5, k) for k in (4096, 11008)}
        tl = synth.target_logits(9300, 1, K_DRAFT, V_LM, 2.0)
        dl = synth.draft_logits_from(tl, 9301, 0.5)
        state["acc"] = (tl, dl, synth.draft_tokens_greedy(dl), synth.draft_tokens_sampled(dl, 9302))
    byts = 0
    for n, k, base, resid, scales in state["packed"]:
        O.linear(O.FMT_NESTED44, n, k, GROUP, base, resid, scales, state["x1"][k], False)
        O.linear(O.FMT_NESTED44, n, k, GROUP, base, resid, scales, state["x5"][k], True)
        byts += draft_bytes(n, k, 1) + verify_bytes(n, k, 5)
    tl, dl, dg, ds = state["acc"]
    O.accept_greedy(dg, tl)
    O.accept_sample(ds, dl, tl, 1.0, synth.seeds_for(0, 1), 0)
    byts += accept_bytes(1, K_DRAFT, V_LM, False) + accept_bytes(1, K_DRAFT, V_LM, True)
    return byts


def cpu_baseline(min_seconds=10.0):
    state = {}
    oracle_sample_step(state)          # packs (untimed) and warms up
    t0 = time.perf_counter()
    byts, steps = 0, 0
    while time.perf_counter() - t0 < min_seconds:
        byts += oracle_sample_step(state)
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": round(byts / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} x (draft M=1 + verify M=5 of the 4096x4096, 11008x4096, 4096x11008 linears, "
                      f"greedy + sampled acceptance B=1 k=4 V=32000), single-threaded C, fp64 accumulation",
            "host_cores_available": len(os.sched_getaffinity(0))}


# ------------------------------------------------------------------ arms
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(x: float, world: int, device=None) -> float:
    """Largest value over the ranks (the job takes as long as its slowest
    replica); a no-op for one process."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: float, steps: int, world: int, t_max_ms: float) -> float:
    """Whole-job throughput: every rank streams bytes_per_step per step (weak
    scaling), the job lasts t_max_ms."""
    return bytes_per_step * steps * world / (t_max_ms * 1e-3) / 1e9


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    state = {}
    oracle_sample_step(state)
    for _ in range(args.warmup):
        oracle_sample_step(state)
    t0 = time.perf_counter()
    byts = sum(oracle_sample_step(state) for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = byts / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": "oracle sample of the round"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "per step: draft M=1 + verify M=5 of three LLaMA-2-7B linear shapes "
                                       "+ greedy and sampled acceptance (B=1, k=4, V=32000)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)          # before the process group: NCCL binds the current device
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from quantized_self_speculative_gb300 import build
    build.build()
    R = Round(device, seed=17 + rank)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        R.run()
    barrier()
    # ---- timed region: K rounds, per-launch events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(K_DRAFT + 3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = cvd.split(",")[local].strip() if cvd else str(local)
    with ClockSampler(smi_index) as clk:
        barrier()
        start.record()
        for s in range(args.steps):
            R.run(ev[s])
        stop.record()
        barrier()
    ms = start.elapsed_time(stop)
    draft_ms = [ev[s][p].elapsed_time(ev[s][p + 1]) for s in range(args.steps) for p in range(K_DRAFT)]
    verify_ms = [ev[s][K_DRAFT].elapsed_time(ev[s][K_DRAFT + 1]) for s in range(args.steps)]
    accept_ms = [ev[s][K_DRAFT + 1].elapsed_time(ev[s][K_DRAFT + 2]) for s in range(args.steps)]
    t_max = reduce_max(ms, world, device)
    # ---- end to end: host activations in, emitted tokens out
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        R.run_e2e()
    e1.record()
    barrier()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device)
    if rank != 0:
        return
    hbm, peak_kind = peaks()
    value = whole_job_gbs(R.bytes_round, args.steps, world, t_max)
    d_avg = statistics.mean(draft_ms)
    v_avg = statistics.mean(verify_ms)
    draft_gbs = R.bytes_draft_pass / (d_avg * 1e-3) / 1e9
    verify_gbs = R.bytes_verify / (v_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "arithmetic": "4-bit / 8-bit codes decoded to fp16, bf16 activations rounded to fp16, fp32 accumulation",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 activations)",
        "config": {"workload": WORKLOAD, "layers": 32, "group": GROUP, "batch": 1, "k": K_DRAFT,
                   "draft_M": 1, "verify_M": K_DRAFT + 1, "vocab": V_LM,
                   "l2": "inputs larger than L2 (6.8 GB packed weights streamed per round)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_peak": round(100 * value / world / hbm, 1),
        "rounds_per_s": round(args.steps * world / (t_max * 1e-3), 2),
        "draft_pass": {"us": round(d_avg * 1e3, 1), "gbs": round(draft_gbs, 1), "bytes": R.bytes_draft_pass},
        "verify_pass": {"us": round(v_avg * 1e3, 1), "gbs": round(verify_gbs, 1), "bytes": R.bytes_verify},
        "accept_round_us": round(statistics.mean(accept_ms) * 1e3, 2),
        "roofline": {"bound": "hbm", "kernel": "draft GEMV (one persistent launch per model pass, M=1)",
                     "achieved": round(draft_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(draft_gbs / hbm, 4), "peak_kind": peak_kind, "traffic": DRAFT_PASS_DRAM_BYTES,
                     "verify_achieved": round(verify_gbs, 1), "verify_frac": round(verify_gbs / hbm, 4),
                     "frac_nominal": round(draft_gbs / NOMINAL_HBM_GBS, 4),
                     "verify_frac_nominal": round(verify_gbs / NOMINAL_HBM_GBS, 4)},
        "clocks": clk.summary(),
        "e2e": {"value": round(whole_job_gbs(R.bytes_round, args.steps, world, e2e_ms), 1), "unit": "GB/s",
                "h2d_bytes_per_step": R.h2d_bytes, "d2h_bytes_per_step": R.d2h_bytes},
        "gpu_launches": R.launches_per_round * args.steps,
        "eq2_time_per_token": eq2_report(d_avg * 1e3, v_avg * 1e3, statistics.mean(accept_ms) * 1e3,
                                         R.time_target_only()),
    }
    if not args.no_extras:
        line["per_linear_llama2_7b"] = per_linear_table(R)
        del R
        torch.cuda.empty_cache()
        RL = RoundLoop(device)
        line["round_measured"] = RL.measure()
        del RL
        torch.cuda.empty_cache()
        line["accept_sweep_B64_V152064"] = accept_sweep(device)
    if args.extras == "full" and not args.no_extras:
        line["config3_llama3_8b_b16_k8"] = config3_sweep(device)
        line["config4_qwen25_7b_tiers"] = config4_sweep(device)
        line["config5_tokens_per_round"] = config5_tokens(device)
        line["kv_nesting_32k"] = kv_sweep(device)
        line["w8a8_llama2_7b"] = a8_sweep(device)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--extras", choices=["quick", "full"], default="full",
                    help="full (default): also the LLaMA-3-8B (M=16/144), Qwen2.5-7B tier and acceptance-sweep "
                         "passes; quick: the LLaMA-2-7B round, per-linear times and acceptance timing only")
    ap.add_argument("--case", default=None,
                    help="profiling workload: draft|verify|draft16|verify144|int4|fp8|fp16|greedy|sample|kv4|kv8")
    ap.add_argument("--layers", type=int, default=8)
    args = ap.parse_args()
    if args.case:
        profile_case(args.case, args.layers)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
