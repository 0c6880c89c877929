#!/usr/bin/env python3
"""Benchmark of the NVFP4 linear path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
AdaLN modulation (when the workload has it) -> global amax -> E4M3 block
scales + E2M1 codes -> block-scaled FP4 GEMM -> bias / residual-gate epilogue,
inputs resident in HBM.  Metric: fused NVFP4 linear TFLOPS (2*M*N*K per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config qkv|tiny|fc1|fc2|attn_out]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Multi-GPU (torchrun, one rank per GPU): independent replicas, each rank runs
the same per-GPU workload (weak scaling, no data-path collective); the timing
is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused NVFP4 linear TFLOPS (% GB300 FP4 peak); act-quant GB/s (% HBM), 1 GPU"
L2_FLUSH_BYTES = 256 << 20
FP4_OVER_BF16 = 6.0   # nominal dense fp4 / bf16 tensor ratio (13.5 / 2.25 PFLOP/s)
DEFAULT_CONFIG = "fc1"
L2_BYTES = 129e6  # GB300 L2; an activation below it is re-read from L2 by the pack pass
CPU_ROWS = {"tiny": 256, "qkv": 256, "fc1": 128, "fc2": 128, "attn_out": 256}  # oracle sample rows per workload
REFERENCE_BUDGET_S = 120.0  # CPU seconds the reference arm's timed steps aim for in total
# DRAM bytes (read + write) per launch of nvfp4_gemm_kernel from one ncu capture
# of the current kernel per workload; None where not captured.
NCU_GEMM_TRAFFIC = {"fc1": 81.63456e6 + 757.145856e6, "fc2": 457.412352e6 + 184.280576e6,
                    "qkv": 30.25152e6 + 99.592704e6, "attn_out": 255.282432e6 + 160.99968e6}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during the timed region."""
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
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- GPU arm

class Problem:
    """Device-resident inputs and outputs of one workload."""

    def __init__(self, name: str, torch, A, data=None):
        import workloads as W
        self.name = name
        d = W.make_inputs(name) if data is None else data
        self.d = d
        self.M, self.N, self.K = d["M"], d["N"], d["K"]
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
        self.x = dev(d["x"])
        self.shift, self.scale, self.gate = f32(d["shift"]), f32(d["scale"]), f32(d["gate"])
        self.resid = None if d["resid"] is None else dev(d["resid"])
        self.bias = dev(d["bias"])
        self.seg_off = [int(v) for v in d["seg_off"]]
        w = dev(d["w"])
        self.wq = A.alloc_nvfp4(self.N, self.K)
        self.ws = A.alloc_workspace(max(self.M, self.N), self.N, self.K, 0)
        A.h3fp4_quantize_weight(w, *self.wq, self.ws)
        del w
        self.aq = A.alloc_nvfp4(self.M, self.K)
        self.out = torch.empty((self.M, self.N), dtype=torch.bfloat16, device="cuda")
        self.flops = 2.0 * self.M * self.N * self.K
        # host copies for the end-to-end leg (pinned)
        self.h_x = torch.empty_like(self.x, device="cpu").pin_memory()
        self.h_x.copy_(self.x)
        self.h_resid = None
        if self.resid is not None:
            self.h_resid = torch.empty_like(self.resid, device="cpu").pin_memory()
            self.h_resid.copy_(self.resid)
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()

    def describe(self):
        wl = self.d["workload"]
        return (f"{wl.name}: X bf16 [{self.M},{self.K}] -> NVFP4 (in-run amax), W NVFP4 [{self.N},{self.K}], "
                f"{wl.description}")

    def quant(self, A):
        A.h3fp4_quantize_act(self.x, *self.aq, self.ws, shift=self.shift, scale=self.scale, seg_off=self.seg_off)

    def quant_given(self, A):
        """Pack pass only: the global scale is the one the last in-run quantisation left."""
        A.h3fp4_quantize_act(self.x, *self.aq, self.ws, shift=self.shift, scale=self.scale, seg_off=self.seg_off,
                             gscale_given=True)

    def gemm(self, A):
        A.h3fp4_linear(self.aq[0], *self.wq, self.out, self.ws, a_sf=self.aq[1], a_gscale=self.aq[2],
                       gate=self.gate, resid=self.resid, bias=self.bias, seg_off=self.seg_off)

    def fused_from_device(self, A, x, resid, out):
        A.h3fp4_linear(x, *self.wq, out, self.ws, shift=self.shift, scale=self.scale, gate=self.gate,
                       resid=resid, bias=self.bias, seg_off=self.seg_off)

    def quant_bytes(self):
        """Algorithmic HBM bytes of the quantiser: the amax pass reads X (2 B per
        element); the pack pass reads X again, writes the codes (0.5 B) and the
        block scales (1/16 B).  The pack pass's read of X counts only where X is
        larger than L2: a smaller activation is still in L2 from the amax pass.
        With a caller-given global scale the pack pass is the only pass and its
        read of X always counts."""
        MK = self.M * self.K
        x_bytes = 2.0 * MK
        reread = x_bytes if x_bytes > L2_BYTES else 0.0
        return {"amax": x_bytes, "pack": reread + 0.5 * MK + MK / 16.0,
                "pack_given": x_bytes + 0.5 * MK + MK / 16.0}

    def gemm_bytes(self):
        MK, NK, MN = self.M * self.K, self.N * self.K, self.M * self.N
        b = 0.5625 * (MK + NK) + 2.0 * MN
        if self.resid is not None:
            b += 2.0 * MN
        return b


def time_fused_quant(torch, A, prob: Problem, steps: int, flush):
    """The quantise-once producer inside the GEMM (h3fp4_linear with
    H3FP4_FUSED_QUANT): per step, the amax pass and the GEMM kernel that packs
    its own activation; and with a caller-given global scale, that kernel
    alone.  CUDA events around the public call, L2 flushed between steps."""
    s = torch.cuda.current_stream()
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    prob.quant(A)
    gs.copy_(prob.aq[2])
    kw = dict(shift=prob.shift, scale=prob.scale, gate=prob.gate, resid=prob.resid, bias=prob.bias,
              seg_off=prob.seg_off, fused=True)
    res = {}
    for key, extra in (("tflops", {}), ("given_scale_tflops", {"a_gscale": gs, "gscale_given": True})):
        call = lambda: A.h3fp4_linear(prob.x, *prob.wq, prob.out, prob.ws, **kw, **extra)
        for _ in range(3):
            flush()
            call()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush()
            ev[i][0].record(s)
            call()
            ev[i][1].record(s)
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
        res[key] = round(prob.flops / (ms * 1e-3) / 1e12, 1)
        res[key.replace("tflops", "ms")] = round(ms, 4)
    A.h3fp4_check(prob.ws)
    res["note"] = ("GEMM kernel quantising its own activation (packer warps, per-tile ready flags); "
                   "in-run scale: amax pass + that kernel")
    return res


def time_mlp_chain(torch, A, steps: int, warmup: int, flush):
    """MLP FC1 -> SwiGLU -> FC2 through the public call, X [32768, 3072] with the
    fc1 recipe and modulation, W1 [24576, 3072] in [gate 128 | up 128] row groups,
    h [32768, 12288], then the fc2 weights, gate and residual. FC1's epilogue
    writes h = bf16(silu(g) * u) and max|h|; FC2 quantises h in one pass with the
    global scale derived from it. For comparison the same FC2 also runs with its
    own two-pass (in-run amax) quantisation of h."""
    import workloads as W
    M = 32768
    d1 = W.swiglu_fc1_inputs(M)
    d2 = W.make_inputs("fc2", M=M, with_x=False)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    N1, K1, N2, K2 = d1["N"], d1["K"], d2["N"], d2["K"]
    x, b1, sh, sc = dev(d1["x"]), dev(d1["bias"]), f32(d1["shift"]), f32(d1["scale"])
    ws1 = A.alloc_workspace(max(M, N1), N1, K1, 0)
    wq1 = A.alloc_nvfp4(N1, K1)
    A.h3fp4_quantize_weight(dev(d1["w"]), *wq1, ws1)
    ws2 = A.alloc_workspace(max(M, N2), N2, K2, 0)
    wq2 = A.alloc_nvfp4(N2, K2)
    A.h3fp4_quantize_weight(dev(d2["w"]), *wq2, ws2)
    b2, g2, r2 = dev(d2["bias"]), f32(d2["gate"]), dev(d2["resid"])
    h = torch.empty((M, N1 // 2), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    gs2 = torch.empty(1, dtype=torch.float32, device="cuda")
    amax = A.h3fp4_ws_out_amax(ws1)
    s = torch.cuda.current_stream()

    def fc1():
        A.h3fp4_linear(x, *wq1, h, ws1, shift=sh, scale=sc, bias=b1, swiglu=True, out_amax=True)

    def fc2(given):
        if given:
            A.h3fp4_gscale_from_amax(amax, gs2)
        A.h3fp4_linear(h, *wq2, out, ws2, a_gscale=gs2 if given else None, gscale_given=given,
                       bias=b2, gate=g2, resid=r2)

    # h straight to NVFP4 from FC1's epilogue under a scale of h fixed beforehand
    # (here the one the amax path derives; a sampler would carry it from a
    # previous step), then FC2 on the codes without any quantisation pass.
    hq = A.alloc_nvfp4(M, N1 // 2)

    def fc1_nvfp4():
        A.h3fp4_linear_swiglu_nvfp4(x, *wq1, hq[0], hq[1], gs2, ws1, shift=sh, scale=sc, bias=b1)

    def fc2_prequant():
        A.h3fp4_linear(hq[0], *wq2, out, ws2, a_sf=hq[1], a_gscale=gs2, bias=b2, gate=g2, resid=r2)

    for _ in range(warmup):
        flush(); fc1(); fc2(True); fc2(False)
    for _ in range(warmup):
        flush(); fc1_nvfp4(); fc2_prequant()
    torch.cuda.synchronize()
    # FC1's GEMM alone (X quantised beforehand) for its tensor roofline
    xq = A.alloc_nvfp4(M, K1)
    A.h3fp4_quantize_act(x, *xq, ws1, shift=sh, scale=sc)
    def fc1_gemm():
        A.h3fp4_linear(xq[0], *wq1, h, ws1, a_sf=xq[1], a_gscale=xq[2], bias=b1, swiglu=True, out_amax=True)
    fc1_gemm()
    t1g = []
    t1, t2, t2b = [], [], []
    tq1, tq2 = [], []
    for _ in range(steps):
        flush()
        eg = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        eg[0].record(s); fc1_gemm(); eg[1].record(s)
        torch.cuda.synchronize()
        t1g.append(eg[0].elapsed_time(eg[1]))
        flush()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(s); fc1(); e[1].record(s); fc2(True); e[2].record(s)
        flush()
        f = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        f[0].record(s); fc2(False); f[1].record(s)
        torch.cuda.synchronize()
        t1.append(e[0].elapsed_time(e[1])); t2.append(e[1].elapsed_time(e[2])); t2b.append(f[0].elapsed_time(f[1]))
        flush()
        q = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        q[0].record(s); fc1_nvfp4(); q[1].record(s); fc2_prequant(); q[2].record(s)
        torch.cuda.synchronize()
        tq1.append(q[0].elapsed_time(q[1])); tq2.append(q[1].elapsed_time(q[2]))
    A.h3fp4_check(ws1)
    A.h3fp4_check(ws2)
    flops = 2.0 * M * K1 * N1 + 2.0 * M * K2 * N2
    step = float(np.mean(t1) + np.mean(t2))
    fc1_gemm_ms = float(np.mean(t1g))
    fc1_gemm_tflops = 2.0 * M * K1 * N1 / (fc1_gemm_ms * 1e-3) / 1e12
    res = {"tflops": round(flops / (step * 1e-3) / 1e12, 1), "ms_per_step": round(step, 4),
           "fc1_swiglu_ms": round(float(np.mean(t1)), 4),
           "fc1_swiglu_gemm_ms": round(fc1_gemm_ms, 4), "fc1_swiglu_gemm_tflops": round(fc1_gemm_tflops, 1),
           "fc2_producer_amax_ms": round(float(np.mean(t2)), 4),
           "fc2_two_pass_ms": round(float(np.mean(t2b)), 4),
           "nvfp4_h": {"ms_per_step": round(float(np.mean(tq1) + np.mean(tq2)), 4),
                       "tflops": round(flops / ((np.mean(tq1) + np.mean(tq2)) * 1e-3) / 1e12, 1),
                       "fc1_swiglu_nvfp4_ms": round(float(np.mean(tq1)), 4),
                       "fc2_prequant_ms": round(float(np.mean(tq2)), 4),
                       "note": "FC1 epilogue writes h as NVFP4 under a scale of h fixed beforehand; FC2 reads the codes"},
           "shape": f"X [{M},{K1}] -> FC1 [{N1},{K1}] + SwiGLU -> h [{M},{N1 // 2}] -> FC2 [{N2},{K2}] + gate/resid"}
    del x, h, out, r2, ws1, ws2, wq1, wq2, hq
    torch.cuda.empty_cache()
    return res


def time_block_graph(torch, A, M: int, steps: int, flush):
    """One transformer block's four projections at M tokens, issued eagerly and
    as a replayed CUDA graph (audio_dit_gb300.graphs): QKV 3072 -> 9216 with the
    prologue, attention output 3072 -> 3072 (two segments, gate, residual),
    FC1 3072 -> 24576 with the SwiGLU producer and its amax, FC2 12288 -> 3072
    on h with the derived scale. Device time per block, L2 flushed before each."""
    from audio_dit_gb300.graphs import GraphBuckets
    g = torch.Generator(device="cuda").manual_seed(1234)
    rn = lambda *sh, std=1.0: torch.randn(*sh, generator=g, device="cuda") * std
    K, NQ, NA, N1, N2 = 3072, 9216, 3072, 24576, 3072
    H = N1 // 2
    wq = {}
    for name, (n, k) in {"qkv": (NQ, K), "att": (NA, K), "fc1": (N1, K), "fc2": (N2, H)}.items():
        wq[name] = A.alloc_nvfp4(n, k)
        wsw = A.alloc_workspace(n, 0, k, A.A_PREQUANT)
        A.h3fp4_quantize_weight(rn(n, k, std=0.02).bfloat16(), *wq[name], wsw)
    b = {n: rn(c, std=0.01).bfloat16() for n, c in [("qkv", NQ), ("att", NA), ("fc1", N1), ("fc2", N2)]}
    sh, sc = rn(1, K, std=0.1), rn(1, K, std=0.1)
    sh2, sc2 = rn(2, K, std=0.1), rn(2, K, std=0.1)
    gate_a, gate_2 = torch.rand(2, NA, generator=g, device="cuda"), torch.rand(1, N2, generator=g, device="cuda")
    x = {n: rn(M, K).bfloat16() for n in ("qkv", "att", "fc1")}
    ra, r2 = rn(M, NA).bfloat16(), rn(M, N2).bfloat16()
    out = {"qkv": torch.empty(M, NQ, dtype=torch.bfloat16, device="cuda"),
           "att": torch.empty(M, NA, dtype=torch.bfloat16, device="cuda"),
           "h": torch.empty(M, H, dtype=torch.bfloat16, device="cuda"),
           "fc2": torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")}
    ws = {n: A.alloc_workspace(M, 0, k, 0) for n, k in [("qkv", K), ("att", K), ("fc1", K), ("fc2", H)]}
    gs2 = torch.empty(1, dtype=torch.float32, device="cuda")
    seg = [0, M - M // 32, M]

    def issue(_key):
        A.h3fp4_linear(x["qkv"], *wq["qkv"], out["qkv"], ws["qkv"], shift=sh, scale=sc, bias=b["qkv"])
        A.h3fp4_linear(x["att"], *wq["att"], out["att"], ws["att"], shift=sh2, scale=sc2, gate=gate_a,
                       resid=ra, bias=b["att"], seg_off=seg)
        A.h3fp4_linear(x["fc1"], *wq["fc1"], out["h"], ws["fc1"], shift=sh, scale=sc, bias=b["fc1"],
                       swiglu=True, out_amax=True)
        A.h3fp4_gscale_from_amax(A.h3fp4_ws_out_amax(ws["fc1"]), gs2)
        A.h3fp4_linear(out["h"], *wq["fc2"], out["fc2"], ws["fc2"], a_gscale=gs2, gscale_given=True,
                       gate=gate_2, resid=r2, bias=b["fc2"])

    graphs = GraphBuckets(issue)
    graphs.capture(M)
    s = torch.cuda.current_stream()
    res = {}
    for mode in ("eager", "graph"):
        ts = []
        for i in range(steps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            if mode == "eager":
                issue(M)
            else:
                graphs.run(M)
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1))
        res[mode + "_ms"] = round(float(np.median(ts)), 4)
    # host time to issue one block (no synchronisation inside the measured region)
    for mode in ("eager", "graph"):
        hs = []
        for i in range(steps + 3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if mode == "eager":
                issue(M)
            else:
                graphs.run(M)
            t1 = time.perf_counter()
            if i >= 3:
                hs.append((t1 - t0) * 1e6)
        res[mode + "_host_issue_us"] = round(float(np.median(hs)), 1)
    torch.cuda.synchronize()
    for w in ws.values():
        A.h3fp4_check(w)
    flops = 2.0 * M * (K * NQ + K * NA + K * N1 + H * N2)
    res["graph_tflops"] = round(flops / (res["graph_ms"] * 1e-3) / 1e12, 1)
    res["launches_per_block"] = "12 kernels + 1 memset"
    return res


def time_m_sweep(torch, A, steps: int, flush, fp4_peak: float):
    """The attention-output shape K = N = 3072 (one segment, gate and residual,
    attn_out value distributions) over M = 1024 ... 65536 tokens: quantiser
    (in-run amax) + GEMM per step, L2 flushed between steps."""
    import workloads as W
    rows = []
    for M in (1024, 2048, 4096, 8192, 16384, 32768, 65536):
        pe = Problem("attn_out", torch, A, data=W.m_sweep_inputs(M))
        q, g, _ = time_device_steps(torch, A, pe, steps, 3, flush)
        qb = pe.quant_bytes()
        gt = pe.flops / (np.mean(g) * 1e-3) / 1e12
        rows.append({"M": M, "tflops": round(pe.flops / (np.mean(q + g) * 1e-3) / 1e12, 1),
                     "gemm_tflops": round(gt, 1), "gemm_frac_fp4_peak": round(gt / fp4_peak, 4),
                     "quant_gbs": round((qb["amax"] + qb["pack"]) / (np.mean(q) * 1e-3) / 1e9, 1),
                     "ms_per_step": round(float(np.mean(q + g)), 4)})
        del pe
        torch.cuda.empty_cache()
    return rows


def time_device_steps(torch, A, prob: Problem, steps: int, warmup: int, flush, given_scale: bool = False):
    """Per-step CUDA events on the launching stream: [quant | gemm], L2 flushed
    between steps. With given_scale the quantisation is the pack pass alone
    (the caller supplies the global scale, as a serving loop with calibrated
    scales would)."""
    s = torch.cuda.current_stream()
    quant = prob.quant_given if given_scale else prob.quant
    prob.quant(A)  # leaves a global scale behind for the given-scale variant
    for _ in range(warmup):
        flush()
        quant(A)
        prob.gemm(A)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0 = time.perf_counter()
    for i in range(steps):
        flush()
        ev[i][0].record(s)
        quant(A)
        ev[i][1].record(s)
        prob.gemm(A)
        ev[i][2].record(s)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    q = np.array([a.elapsed_time(b) for a, b, _ in ev])
    g = np.array([b.elapsed_time(c) for _, b, c in ev])
    A.h3fp4_check(prob.ws)
    return q, g, wall


def time_e2e(torch, A, prob: Problem, steps: int, warmup: int, copy_streams: int = 1):
    """Public API end to end: each step copies its X (+R) from pinned host memory,
    runs the fused h3fp4_linear and copies its bf16 output back to pinned host
    memory. Copies in, compute and copies out run on separate streams with two
    buffer sets, so one step's output copy overlaps the next step's input copy
    and compute (a serving pipeline); each copy is split by rows over
    `copy_streams` streams so that several copy engines share it. Event
    dependencies keep every buffer from being reused before its previous step
    is done with it. The timed region spans the first input copy to the last
    output copy."""
    main = torch.cuda.current_stream()
    s_comp = torch.cuda.Stream()
    ins = [torch.cuda.Stream() for _ in range(copy_streams)]
    outs_s = [torch.cuda.Stream() for _ in range(copy_streams)]
    nb = 2
    xs = [torch.empty_like(prob.x) for _ in range(nb)]
    rs = [None if prob.resid is None else torch.empty_like(prob.resid) for _ in range(nb)]
    outs = [torch.empty_like(prob.out) for _ in range(nb)]
    h_outs = [prob.h_out] + [torch.empty_like(prob.h_out).pin_memory() for _ in range(nb - 1)]
    ev = lambda: torch.cuda.Event()
    in_done = [[ev() for _ in range(copy_streams)] for _ in range(nb)]
    comp_done = [ev() for _ in range(nb)]
    out_done = [[ev() for _ in range(copy_streams)] for _ in range(nb)]
    used = [False] * nb
    rows = lambda t, c: t.narrow(0, c * t.shape[0] // copy_streams,
                                 (c + 1) * t.shape[0] // copy_streams - c * t.shape[0] // copy_streams)

    def step(i):
        b = i % nb
        for c, st in enumerate(ins):
            with torch.cuda.stream(st):
                if used[b]:
                    st.wait_event(comp_done[b])          # step i-2 has consumed xs[b] / rs[b]
                rows(xs[b], c).copy_(rows(prob.h_x, c), non_blocking=True)
                if rs[b] is not None:
                    rows(rs[b], c).copy_(rows(prob.h_resid, c), non_blocking=True)
                in_done[b][c].record(st)
        with torch.cuda.stream(s_comp):
            for c in range(copy_streams):
                s_comp.wait_event(in_done[b][c])
                if used[b]:
                    s_comp.wait_event(out_done[b][c])    # step i-2's output copy has read outs[b]
            prob.fused_from_device(A, xs[b], rs[b], outs[b])
            comp_done[b].record(s_comp)
        for c, st in enumerate(outs_s):
            with torch.cuda.stream(st):
                st.wait_event(comp_done[b])
                rows(h_outs[b], c).copy_(rows(outs[b], c), non_blocking=True)
                out_done[b][c].record(st)
        used[b] = True

    streams = [s_comp] + ins + outs_s
    for st in streams:
        st.wait_stream(main)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for st in streams:
        st.wait_event(e0)
    for i in range(steps):
        step(warmup + i)
    for st in streams:
        main.wait_stream(st)
    e1.record(main)
    torch.cuda.synchronize()
    A.h3fp4_check(prob.ws)
    ms = e0.elapsed_time(e1) / steps
    h2d = prob.h_x.numel() * 2 + (0 if prob.h_resid is None else prob.h_resid.numel() * 2)
    d2h = prob.h_out.numel() * 2
    return ms, h2d, d2h


class OracleSample:
    """The CPU oracle, as it stands, on the first rows of a workload: quantise
    those rows of X (their own amax), then every output of those rows in
    float64 (GEMM + epilogue). W is quantised once beforehand (offline, as the
    method quantises weights); it is not part of a step."""

    def __init__(self, name: str, rows: int):
        import oracle
        import workloads as W
        self.oracle = oracle
        self.d = W.make_inputs(name, M=rows)
        t0 = time.perf_counter()
        self.w = oracle.quantize(self.d["w"])
        self.quantize_w_s = time.perf_counter() - t0
        self.last_split = (0.0, 0.0)

    def step(self, rows: int):
        """Returns (TFLOP/s, seconds) for the first `rows` rows; the split
        (quantise X, GEMM + epilogue) in seconds is kept in last_split."""
        d = self.d
        seg = np.minimum(d["seg_off"], rows)
        t0 = time.perf_counter()
        a = self.oracle.quantize(d["x"][:rows], d["shift"], d["scale"], seg)
        t1 = time.perf_counter()
        self.oracle.linear_full(a, self.w, rows, d["N"], d["K"], bias=d["bias"], gate=d["gate"],
                                resid=None if d["resid"] is None else d["resid"][:rows], seg_off=seg)
        t2 = time.perf_counter()
        self.last_split = (t1 - t0, t2 - t1)
        return 2.0 * rows * d["N"] * d["K"] / (t2 - t0) / 1e12, t2 - t0


def oracle_sample(name: str, rows: int):
    """One timed oracle step on the first `rows` rows (see OracleSample).
    Returns (TFLOP/s, seconds, threads, {quantise_x_s, gemm_epilogue_s, quantise_w_s})."""
    s = OracleSample(name, rows)
    tf, dt = s.step(rows)
    split = {"quantise_x_s": round(s.last_split[0], 3), "gemm_epilogue_s": round(s.last_split[1], 3),
             "quantise_w_s": round(s.quantize_w_s, 3)}
    return tf, dt, s.oracle.num_threads(), split


def run_gpu(args):
    import torch
    import audio_dit_gb300 as A
    from audio_dit_gb300 import build as B

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or not os.path.exists(A.library_path()):
        B.build()
    if dist is not None:
        dist.barrier()
    A.load_library()
    peaks = load_peaks()

    prob = Problem(args.config, torch, A)
    # L2 flush between steps (untimed): write a buffer larger than L2, then read
    # another one, so the timed kernels start with none of their inputs cached
    # and without the flush's own dirty lines still waiting to be written back.
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_sum = torch.empty((), dtype=torch.float32, device="cuda")

    def flush():
        flush_buf.fill_(1)
        torch.sum(flush_rd, dim=0, out=flush_sum)

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        q, g, wall = time_device_steps(torch, A, prob, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    step_ms = float(np.mean(q + g))
    if dist is not None:
        t = torch.tensor([step_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
        dist.barrier()
    e2e_ms, h2d, d2h = time_e2e(torch, A, prob, max(3, args.steps // 2), args.warmup)
    if dist is not None:
        t = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    value = world * prob.flops / (step_ms * 1e-3) / 1e12
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    mma_peak = A.h3fp4_measure_fp4_peak(prob.ws, 20000) if rank == 0 else None
    pair_peak = A.h3fp4_measure_fp4_pair_peak(prob.ws, 20000) if rank == 0 else None
    # every NVFP4 (kind::mxf4nvf4, scale_vec::4X) MMA form, back to back, operands on chip
    forms = ({A.MMA_FORMS[f]: round(A.h3fp4_measure_fp4_form(prob.ws, f, 20000), 1) for f in sorted(A.MMA_FORMS)}
             if rank == 0 else None)
    gemm_ms = float(np.mean(g))
    gemm_tflops = prob.flops / (gemm_ms * 1e-3) / 1e12
    qb = prob.quant_bytes()
    quant_ms = float(np.mean(q))
    quant_gbs = (qb["amax"] + qb["pack"]) / (quant_ms * 1e-3) / 1e9

    given = fused_q = None
    if rank == 0:
        qg, gg, _ = time_device_steps(torch, A, prob, max(5, min(500, args.steps // 4)), 3, flush, given_scale=True)
        given = {"tflops": round(prob.flops / (np.mean(qg + gg) * 1e-3) / 1e12, 1),
                 "quant_ms": round(float(np.mean(qg)), 5),
                 "quant_gbs": round(qb["pack_given"] / (np.mean(qg) * 1e-3) / 1e9, 1),
                 "note": "global scale supplied by the caller: pack pass + GEMM"}
        fused_q = time_fused_quant(torch, A, prob, max(5, min(200, args.steps // 4)), flush)

    extra = {}
    if rank == 0 and not args.no_extra:
        for name in [c for c in ["tiny", "qkv", "fc1", "fc2", "attn_out"] if c != args.config]:
            try:
                pe = Problem(name, torch, A)
                qe, ge, _ = time_device_steps(torch, A, pe, max(5, min(200, args.steps // 4)), 3, flush)
                qge, gge, _ = time_device_steps(torch, A, pe, max(5, min(200, args.steps // 4)), 3, flush,
                                                given_scale=True)
                qbe = pe.quant_bytes()
                extra[name] = {
                    "tflops": round(pe.flops / (np.mean(qe + ge) * 1e-3) / 1e12, 1),
                    "gemm_tflops": round(pe.flops / (np.mean(ge) * 1e-3) / 1e12, 1),
                    "gemm_frac_fp4_peak": round(pe.flops / (np.mean(ge) * 1e-3) / 1e12 / fp4_peak, 4),
                    "quant_gbs": round((qbe["amax"] + qbe["pack"]) / (np.mean(qe) * 1e-3) / 1e9, 1),
                    "ms_per_step": round(float(np.mean(qe + ge)), 4),
                    "given_scale_tflops": round(pe.flops / (np.mean(qge + gge) * 1e-3) / 1e12, 1),
                    "given_scale_quant_gbs": round(qbe["pack_given"] / (np.mean(qge) * 1e-3) / 1e9, 1),
                }
                if name != "tiny":
                    extra[name]["fused_quant"] = time_fused_quant(torch, A, pe, max(5, min(100, args.steps // 8)),
                                                                  flush)
                del pe
                torch.cuda.empty_cache()
            except Exception as e:  # a failing extra config must not hide the headline
                extra[name] = {"error": repr(e)[:200]}
        try:
            extra["m_sweep"] = time_m_sweep(torch, A, max(5, min(100, args.steps // 20)), flush, fp4_peak)
        except Exception as e:
            extra["m_sweep"] = {"error": repr(e)[:200]}
        try:
            extra["mlp_swiglu"] = time_mlp_chain(torch, A, max(3, min(50, args.steps // 40)), 3, flush)
            extra["mlp_swiglu"]["fc1_swiglu_gemm_frac_fp4_peak"] = round(
                extra["mlp_swiglu"]["fc1_swiglu_gemm_tflops"] / fp4_peak, 4)
        except Exception as e:
            extra["mlp_swiglu"] = {"error": repr(e)[:200]}
        for bm in (1024, 8192):
            try:
                extra[f"block_graph_m{bm}"] = time_block_graph(torch, A, bm, max(3, min(30, args.steps // 60)), flush)
                torch.cuda.empty_cache()
            except Exception as e:
                extra[f"block_graph_m{bm}"] = {"error": repr(e)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def cpu_line(name, rows):
            tf, dt, cores, split = oracle_sample(name, rows)
            wl = W.WORKLOADS[name]
            return {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "split": split,
                    "sample": f"first {rows} rows of {name} (own amax), all {rows}x{wl.N} outputs in "
                              f"float64, W quantised once beforehand; {dt:.1f} s"}
        import workloads as W
        cpu = cpu_line(args.config, args.cpu_rows or CPU_ROWS[args.config])
        if not args.no_extra:
            for name in [c for c in CPU_ROWS if c != args.config]:
                if name in extra and "error" not in extra[name]:
                    try:
                        extra[name]["cpu_baseline"] = cpu_line(name, CPU_ROWS[name])
                    except Exception as e:
                        extra[name]["cpu_baseline"] = {"error": repr(e)[:200]}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOPS",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(step_ms, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x e2m1, e4m3 block scales, fp32 accumulate)",
            "data": "synthetic (seeded, shapes/distributions of the workload set)",
            "config": {"workload": prob.describe(), "M": prob.M, "N": prob.N, "K": prob.K,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB written, then {L2_FLUSH_BYTES >> 20} MiB read; untimed)",
                       "global_scale": "computed in-run (amax pass)"},
            "e2e": {"value": round(world * prob.flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOPS",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": 3 * args.steps,
            "roofline": {"bound": "tensor", "kernel": "nvfp4_gemm_kernel",
                         "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                         "frac": round(gemm_tflops / fp4_peak, 4),
                         "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} x nominal fp4/bf16 6",
                         "measured_mma_peak": round(mma_peak, 1) if mma_peak else None,
                         "frac_of_measured_mma_peak": round(gemm_tflops / mma_peak, 4) if mma_peak else None,
                         "measured_pair_mma_peak": round(pair_peak, 1) if pair_peak else None,
                         "frac_of_measured_pair_mma_peak": round(gemm_tflops / pair_peak, 4) if pair_peak else None,
                         "measured_mma_forms": forms,
                         "traffic": NCU_GEMM_TRAFFIC.get(args.config), "algorithmic_bytes": prob.gemm_bytes()},
            "quant": {"gbs": round(quant_gbs, 1), "peak_gbs": peaks["hbm_gbs"],
                      "frac": round(quant_gbs / peaks["hbm_gbs"], 4), "ms": round(quant_ms, 5),
                      "bytes": "amax read 2 B/elem + pack re-read of X 2 B/elem (only where X exceeds L2) "
                               "+ codes 0.5 + scales 1/16 B/elem",
                      "algorithmic_bytes": qb["amax"] + qb["pack"]},
            "gemm_ms": round(gemm_ms, 5),
            "timing": {"gemm_ms_median": round(float(np.median(g)), 5), "gemm_ms_best": round(float(np.min(g)), 5),
                       "quant_ms_median": round(float(np.median(q)), 5), "quant_ms_best": round(float(np.min(q)), 5),
                       "step_ms_median": round(float(np.median(q + g)), 5),
                       "step_ms_best": round(float(np.min(q + g)), 5),
                       "note": "value, gemm_ms and quant.ms are means over the timed steps"},
            "clocks": clk.summary(),
            "wall_s_timed": round(wall, 3),
        }
        if given:
            line["given_scale"] = given
        if fused_q is not None:
            line["fused_quant"] = fused_q
        if extra:
            line["also"] = extra
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- reference arm (oracle)

def run_reference(args):
    """The oracle as the reference arm, timed on the host cores. Each step is a
    bounded sample of the workload: its rows per step are chosen from the
    warm-up's time per row so that all --steps steps take about
    REFERENCE_BUDGET_S seconds (at most 256 rows per step)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import workloads as W
    import oracle
    oracle.build()
    max_rows = args.cpu_rows or CPU_ROWS[args.config]
    sample = OracleSample(args.config, max_rows)
    per_row = []
    for _ in range(args.warmup):
        _, dt = sample.step(8)
        per_row.append(dt / 8)
    per_row_s = float(np.median(per_row)) if per_row else 0.03
    rows = int(max(1, min(max_rows, REFERENCE_BUDGET_S / max(1, args.steps) / max(per_row_s, 1e-6))))
    vals, times = [], []
    for _ in range(args.steps):
        tf, dt = sample.step(rows)
        vals.append(tf)
        times.append(dt)
    wl = W.WORKLOADS[args.config]
    v = float(2.0 * rows * wl.N * wl.K * len(times) / sum(times) / 1e12)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": float(np.mean(times)) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (oracle: fp32 quantiser, float64 GEMM)",
        "data": "synthetic (seeded, shapes/distributions of the workload set)",
        "config": {"workload": f"{wl.name}: first {rows} rows of X [{wl.M},{wl.K}] per step, W [{wl.N},{wl.K}]",
                   "M": rows, "N": wl.N, "K": wl.K},
        "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{rows} rows of {wl.name} per step (quantise + float64 GEMM/epilogue; "
                                   f"W quantised once beforehand)"},
        "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=["tiny", "qkv", "fc1", "fc2", "attn_out"])
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle sample rows (0: per-workload default)")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
