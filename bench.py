#!/usr/bin/env python3
"""Benchmark of the hot path on GB300: one training step of the last
transformer layer plus its tied-embedding LM head.

Step (all on the GPU, through the C ABI):
  y = layer_fwd(x)                                   (GQA 32q/8kv x 128, SwiGLU 11008,
                                                      causal, Pre-LN, B2 S4096 H4096)
  loss, d_y, d_E = vocab_ce_fwd_bwd(y, E, targets)   (V 128256, chunks of 16032)
  d_x, d_W = layer_bwd(d_y)

`value` = model TFLOP/s of the step (2MNK per GEMM, attention 4*B*nq*d*pairs,
backward 2x forward, recompute not counted), inputs resident in HBM. `e2e`
times the same step with x and targets copied from pinned host memory each
step and the mean loss read back. `roofline` is the tcgen05 GEMM kernel,
timed live with CUDA events on its stream inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica (no collective on the
data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from megatron_transformer_layer_fwd_gb300.inputs import (CE_WORKLOADS, WORKLOADS, CEShape,  # noqa: E402
                                                         ce_flops, ce_inputs, ce_stream_bytes,
                                                         layer_flops, layer_inputs)

METRIC = "layer fwd+bwd TFLOP/s and tokens/s (bf16) + vocab-CE GB/s, % of roofline"
LAYER = "bf16_gqa_swiglu_b2s4096h4096"
CE = "bf16_ce_t8192h4096v128256"
WORKLOAD = (f"{LAYER} -> {CE}: layer fwd, tied-embedding CE fwd+bwd on the layer output, "
            "layer bwd from the CE gradient")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 200 ms)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", self.index, "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def smi_index() -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    first = vis.split(",")[0].strip() if vis else ""
    if first.isdigit():
        return first
    return os.environ.get("LOCAL_RANK", "0")


# ------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle

class OracleSample:
    """The float64 oracle on a bounded sample of the same workload: the layer
    fwd+bwd at full width (hidden, heads, ffn) with 128 tokens, and the CE
    fwd+bwd of 32 tokens against the full vocabulary. Inputs are drawn once."""

    SEQ, CE_TOKENS = 128, 32

    def __init__(self):
        import oracle
        self.oracle = oracle
        self.shape = WORKLOADS[LAYER].replace(batch=1, seq=self.SEQ)
        arr = layer_inputs(self.shape, seed=0)
        self.w = {k: arr[k] for k in ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2",
                                      "ln1_g", "ln1_b", "ln2_g", "ln2_b")}
        self.x = arr["x"]
        self.dy = np.full((self.shape.tokens, self.shape.hidden),
                          1.0 / (self.shape.tokens * self.shape.hidden))
        self.ce = CE_WORKLOADS[CE]
        rng = np.random.default_rng(0)
        n = self.CE_TOKENS
        self.hid = rng.standard_normal((n, self.ce.hidden))
        self.emb = rng.standard_normal((self.ce.vocab, self.ce.hidden), dtype=np.float32) * 0.02
        self.emb = self.emb.astype(np.float64)
        self.tg = rng.integers(0, self.ce.vocab, n)
        self.flops = layer_flops(self.shape)["total"] + 3 * 2.0 * n * self.ce.vocab * self.ce.hidden
        self.desc = (f"layer fwd+bwd at B1 S{self.SEQ} (full hidden/heads/ffn of {LAYER}) + CE "
                     f"fwd+bwd for {n} tokens x the full {self.ce.vocab}-entry vocabulary, "
                     "float64 numpy")

    def run_once(self) -> float:
        """One sample; returns seconds."""
        o = self.oracle
        t0 = time.perf_counter()
        _, c = o.block_fwd(self.shape, self.w, self.x)
        o.block_bwd(self.shape, self.w, c, self.dy)
        n = self.CE_TOKENS
        _, lse, _ = o.ce_full(self.hid, self.emb, self.tg, row_block=n)
        o.ce_grads(self.hid, self.emb, self.tg, lse, 1.0 / n, row_block=n)
        return time.perf_counter() - t0

    def timed(self, budget_s: float) -> dict:
        t, reps = 0.0, 0
        while reps == 0 or (t < budget_s and reps < 50):
            t += self.run_once()
            reps += 1
        return {"value": reps * self.flops / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                "kind": "oracle", "seconds": round(t, 2), "sample": f"{reps} x [{self.desc}]"}


# ------------------------------------------------------------ our arm

def traffic_record(kernel_src: str, kind: str) -> float | None:
    """Per-launch DRAM bytes (read + write) of a kernel kind from the committed
    ncu summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    if d.get("source_sha256_16") != h:
        return None
    return d.get("kinds", {}).get(kind, {}).get("bytes_per_launch")


def run_ours(args, world, rank, local):
    import torch
    from megatron_transformer_layer_fwd_gb300 import build, mgb
    from megatron_transformer_layer_fwd_gb300.runner import CERunner, LayerRunner, to_device

    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = WORKLOADS[LAYER]
    ce = CE_WORKLOADS[CE]
    arr = layer_inputs(shape, seed=rank)
    layer = LayerRunner(shape, arr, device=dev)
    cin = ce_inputs(ce, seed=rank)
    emb = to_device(cin["emb"], torch.bfloat16, dev)
    targets = torch.from_numpy(cin["targets"]).to(dev)
    del cin, arr
    # the step's stream outranks the library's side streams (lowest priority):
    # when SMs free up, the critical path's pending blocks start first
    torch.cuda.synchronize(dev)  # inputs copied on the default stream are in place
    stream = torch.cuda.Stream(dev, priority=-1)
    torch.cuda.set_stream(stream)
    # the CE's weight gradient d_emb (its last token block) runs on its own
    # stream, beside the layer backward (which needs only d_hidden); each step
    # ends by joining it
    emb_stream = torch.cuda.Stream(dev)
    cer = CERunner(ce.tokens, ce.hidden, ce.vocab, ce.chunk, layer.y, emb, targets,
                   mode=mgb.MGB_CE_BLOCKED, emb_stream=emb_stream, token_block=args.token_block)

    def make_step(c):
        def step():
            layer.fwd(stream)
            c.run(stream)
            layer.bwd(c.d_hidden, stream)
            stream.wait_stream(emb_stream)
        return step

    step = make_step(cer)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if mgb.mgb_device_status(stream) != mgb.MGB_OK:
        raise RuntimeError("device error during warm-up")

    # ---- timed region: inputs resident in HBM (working set >> L2)
    mgb.mgb_profile_reset()
    mgb.mgb_profile_enable(True)
    clocks = ClockSampler(smi_index())
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    n0 = mgb.mgb_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    launches = (mgb.mgb_launch_count() - n0) // args.steps
    mgb.mgb_profile_enable(False)
    prof = mgb.mgb_profile_read()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(world, ms)
    if mgb.mgb_device_status(stream) != mgb.MGB_OK:
        raise RuntimeError("device error during the timed region")

    # ---- the layer alone (fwd + bwd from the CE gradient of the last step)
    barrier(world)
    torch.cuda.synchronize(dev)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(args.steps):
        layer.fwd(stream)
        layer.bwd(cer.d_hidden, stream)
    l1.record(stream)
    torch.cuda.synchronize(dev)
    layer_ms = max_over_ranks(world, l0.elapsed_time(l1) / args.steps)

    # ---- end to end through host buffers: every step copies x and the
    # targets from pinned host memory with the library's copy call and reads
    # the mean loss back; device-only steps are interleaved with them (each
    # step between its own events), so that clock drift under the power cap
    # falls on both alike and the difference is the copies' cost
    x_host = layer.x.cpu().pin_memory()
    t_host = targets.cpu().pin_memory()
    loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
    h2d = layer.x.numel() * layer.x.element_size() + targets.numel() * 4

    def e2e_step():
        mgb.mgb_memcpy_async(layer.x, x_host, layer.x.numel() * layer.x.element_size(), stream)
        mgb.mgb_memcpy_async(targets, t_host, targets.numel() * 4, stream)
        step()
        mgb.mgb_memcpy_async(loss_host, cer.loss_mean, 4, stream)

    barrier(world)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(2 * args.steps)]
    for i, (a, b) in enumerate(ev):
        a.record(stream)
        (e2e_step if i % 2 == 0 else step)()
        b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_times = [a.elapsed_time(b) for a, b in ev[0::2]]
    dev_times = [a.elapsed_time(b) for a, b in ev[1::2]]
    e2e_ms = max_over_ranks(world, statistics.median(e2e_times))
    dev_inter_ms = max_over_ranks(world, statistics.median(dev_times))

    lf, cf = layer_flops(shape), ce_flops(ce)
    step_flops = lf["total"] + cf["total"]
    value = world * step_flops / (ms / 1e3) / 1e12
    peaks = load_peaks()
    tb = cer.token_block
    # Dominant kernel: the CE logits GEMM (per token block, every vocab chunk
    # in one launch, statistics epilogue storing the block's logits), the
    # longest kernel of the step that runs alone on its stream (the two CE
    # gradient products run side by side and are timed as one phase below).
    # Algorithmic FLOPs per launch (2*rows*V*H) / mean launch time from the
    # library's events on the launching stream inside the timed region.
    ce_kind_flops = 2.0 * ce.tokens * ce.vocab * ce.hidden  # per kind per step
    d_ms, d_n = prof["gemm_tc_ce_logits"]
    d_flops = ce_kind_flops * args.steps / d_n if d_n else 0.0
    d_tflops = d_flops / (d_ms / d_n / 1e3) / 1e12 if d_n else None
    traffic = traffic_record(os.path.join(ROOT, "megatron_transformer_layer_fwd_gb300", "csrc",
                                          "gemm_tc.cu"), f"gemm_tc_ce_logits_tb{tb}")
    roofline = {"kernel": f"gemm_tc_pair_kernel, CE logits per token block {tb}x{ce.vocab}x"
                          f"{ce.hidden} (all vocab chunks of {ce.chunk} in one launch; statistics "
                          "epilogue storing the block's bf16 logits)",
                "bound": "tensor", "achieved": round(d_tflops, 1) if d_tflops else None,
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": round(d_tflops / peaks["bf16_tflops_sustained"], 4) if d_tflops else None,
                "peak_source": f"{peaks['source']} bf16_tflops_sustained (kernel inside a long step)",
                "flops_per_launch": d_flops, "launches_per_step": d_n / args.steps,
                "avg_launch_ms": round(d_ms / d_n, 4) if d_n else None,
                "traffic": traffic}
    # the block's d_hidden (split-K) and d_emb (float32 reduce-add) products,
    # side by side: FLOPs of both / the phase from fork to join
    p_ms, p_n = prof.get("stage_ce_products", (0.0, 0))
    roofline_ce_products = {
        "kernel": "gemm_tc_ce_dgrad (G E, split over K) beside gemm_tc_ce_wgrad (G^T hidden, "
                  "float32 TMA reduce-add) per token block, fork to join",
        "bound": "tensor", "unit": "TFLOP/s", "peak": peaks["bf16_tflops_sustained"],
        "phases_per_step": p_n / args.steps,
        "avg_phase_ms": round(p_ms / p_n, 4) if p_n else None,
        "note": "the last block's d_emb runs on the caller's stream beside the layer backward "
                "and is not inside its phase"}
    if p_n:
        # the phases cover both products of every block but the last one's
        # d_emb: flops = 2 kinds x per-block share for blocks before the last,
        # d_hidden only for the last
        nb = p_n // args.steps
        per_block = ce_kind_flops / nb
        fl = (2 * (nb - 1) + 1) * per_block * args.steps
        roofline_ce_products["achieved"] = round(fl / (p_ms / 1e3) / 1e12, 1)
        roofline_ce_products["frac"] = round(roofline_ce_products["achieved"] /
                                             peaks["bf16_tflops_sustained"], 4)
    # all tcgen05 GEMM work of the step (2MNK each, none recomputed)
    gemm_flops_step = 3 * lf["gemm_fwd"] + 3 * 2.0 * ce.tokens * ce.vocab * ce.hidden
    gemm_kinds = ("gemm_tc_fwd", "gemm_tc_dgrad", "gemm_tc_wgrad", "gemm_tc_ce_logits",
                  "gemm_tc_ce_dgrad", "gemm_tc_ce_wgrad")
    gemm_all = {"tflop_per_step": round(gemm_flops_step / 1e12, 3),
                "share_of_step_flops": round(gemm_flops_step / step_flops, 4),
                "launches_per_step": sum(prof[k][1] for k in gemm_kinds) / args.steps}
    # the HBM-bound CE kernel of the step: ce_grad over each token block's
    # logits [rows, V], read and rewritten in place with G (4 B per logit)
    rg_ms, rg_n = prof.get("ce_grad", (0.0, 0))
    rg_bytes = 4.0 * ce.tokens * ce.vocab * args.steps
    rg_gbs = rg_bytes / (rg_ms / 1e3) / 1e9 if rg_ms > 0 else None
    roofline_ce = {
        "kernel": f"ce_grad over each token block's logits ({tb} x {ce.vocab}, in place)",
        "bound": "hbm", "achieved": round(rg_gbs, 1) if rg_gbs else None, "peak": peaks["hbm_gbs"],
        "unit": "GB/s", "frac": round(rg_gbs / peaks["hbm_gbs"], 4) if rg_gbs else None,
        "peak_source": f"{peaks['source']} hbm_gbs",
        "bytes_per_launch": 4.0 * tb * ce.vocab, "launches_per_step": rg_n / args.steps,
        "avg_launch_ms": round(rg_ms / rg_n, 4) if rg_n > 0 else None}
    # The same step with the resident-logits CE (the whole [T, V] logits held:
    # outside the pages' memory bound), for comparison; a few steps after the
    # timed region.
    res = CERunner(ce.tokens, ce.hidden, ce.vocab, ce.chunk, layer.y, emb, targets,
                   mode=mgb.MGB_CE_RESIDENT, emb_stream=emb_stream)
    rstep = make_step(res)
    for _ in range(2):
        rstep()
    torch.cuda.synchronize(dev)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r_steps = max(3, args.steps // 3)
    r0.record(stream)
    for _ in range(r_steps):
        rstep()
    r1.record(stream)
    torch.cuda.synchronize(dev)
    res_ms = r0.elapsed_time(r1) / r_steps
    step_resident = {"ms_per_step": round(res_ms, 4),
                     "tflops": round(world * step_flops / (res_ms / 1e3) / 1e12, 2),
                     "ce_workspace_gb": round(mgb.mgb_vocab_ce_sizes(mgb.ce_desc(
                         ce.tokens, ce.hidden, ce.vocab, ce.chunk, 1.0 / ce.tokens,
                         mgb.MGB_CE_RESIDENT)) / 1e9, 3),
                     "note": "same step with MGB_CE_RESIDENT (whole [T, V] logits kept); "
                             "outside the pages' memory bound, for comparison only"}
    # the same step with MGB_CE_FUSED: vocab chunks through the logits GEMM's
    # epilogue, no logits stored at all, the logits recomputed for the gradient
    fus = CERunner(ce.tokens, ce.hidden, ce.vocab, ce.chunk, layer.y, emb, targets,
                   mode=mgb.MGB_CE_FUSED, emb_stream=emb_stream)
    fstep = make_step(fus)
    for _ in range(2):
        fstep()
    torch.cuda.synchronize(dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(r_steps):
        fstep()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    fus_ms = f0.elapsed_time(f1) / r_steps
    step_fused = {"ms_per_step": round(fus_ms, 4),
                  "tflops": round(world * step_flops / (fus_ms / 1e3) / 1e12, 2),
                  "ce_workspace_gb": round(mgb.mgb_vocab_ce_sizes(mgb.ce_desc(
                      ce.tokens, ce.hidden, ce.vocab, ce.chunk, 1.0 / ce.tokens,
                      mgb.MGB_CE_FUSED)) / 1e9, 3),
                  "note": "same step with MGB_CE_FUSED (per-chunk statistics and G in the "
                          "logits GEMM's epilogue, no logits stored; the logits are computed "
                          "twice, so its TFLOP/s counts the step's work, not the recompute)"}
    del fus
    breakdown = {k: round(v[0] / args.steps, 4) for k, v in prof.items() if v[1] > 0}
    # page 1's sequence sweep on the causal workloads (B 8, H 2048, 16 x 128, F
    # 8192): the Attention / FFN / Backward stages per length (library events)
    del res
    sweep = None if args.no_sweep else stage_sweep(stream)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded: x~N(0,1), W~N(0,0.02^2), biases 0, LN gamma 1 beta 0, "
                "E~N(0,0.02^2), targets~U[0,V))",
        "config": {"workload": WORKLOAD, "tokens_per_step": shape.tokens,
                   "l2": "inputs larger than L2 (weights 0.35 GB + embedding 1.05 GB + activations)",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * shape.tokens / (ms / 1e3), 1),
        "layer_fwd_bwd": {"ms": round(layer_ms, 4),
                          "tflops": round(world * lf["total"] / (layer_ms / 1e3) / 1e12, 1),
                          "tokens_per_s": round(world * shape.tokens / (layer_ms / 1e3), 1),
                          "frac_of_nominal_2250": round(lf["total"] / (layer_ms / 1e3) / 2.25e15, 4),
                          "frac_of_measured_burst": round(
                              lf["total"] / (layer_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4)},
        "step_tflop": round(step_flops / 1e12, 4),
        "clocks": clk,
        "e2e": {"value": round(world * step_flops / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4,
                "how": "median of steps that copy x and the targets from pinned host memory "
                       "(mgb_memcpy_async) and read the mean loss back, interleaved with "
                       "device-only steps",
                "device_only_interleaved_ms": round(dev_inter_ms, 4),
                "copy_overhead_ms": round(e2e_ms - dev_inter_ms, 4)},
        "gpu_launches": int(launches),
        "roofline": roofline,
        "roofline_ce_products": roofline_ce_products,
        "roofline_ce": roofline_ce,
        "ce": {"mode": "MGB_CE_BLOCKED", "token_block": tb,
               "workspace_gb": round(cer.ws.numel() / 1e9, 3),
               "full_logits_gb": round(2.0 * ce.tokens * ce.vocab / 1e9, 3)},
        "step_resident_ce": step_resident,
        "step_fused_ce": step_fused,
        "seq_sweep": sweep,
        "gemm_all_launches": gemm_all,
        "kernel_ms_per_step": breakdown,
        "kernel_ms_note": "per kind, the span between library CUDA events on the launching "
                          "stream; kernels on the side streams run beside others, so the spans "
                          "overlap and do not add up to ms_per_step",
    }
    return out


def stage_sweep(stream, steps: int = 5, warmup: int = 3) -> dict:
    """Layer fwd+bwd on the causal workloads at S = 128 ... 2048 (batch 8):
    per length the whole layer and page 1's three stages (Attention: LN1, QKV,
    attention, projection; FFN: LN2, fc1, fc2; Backward), and the growth per
    doubling of S against the work's (attention core 4x, FFN 2x)."""
    import torch
    from megatron_transformer_layer_fwd_gb300.runner import LayerRunner
    out = {"workloads": "bf16_causal_b8s{S}h2048", "seq": [], "layer_ms": [],
           "stage_ms": {"attention": [], "ffn": [], "backward": []}, "attention_core_ms": []}
    for seq in (128, 256, 512, 1024, 2048):
        shape = WORKLOADS[f"bf16_causal_b8s{seq}h2048"]
        r = LayerRunner(shape, layer_inputs(shape, seed=0))
        dy = torch.full_like(r.x, 1.0 / (shape.tokens * shape.hidden))

        def fb():
            r.fwd(stream)
            r.bwd(dy, stream)
        ms, prof = _time_loop(fb, steps, warmup, stream)
        out["seq"].append(seq)
        out["layer_ms"].append(round(ms, 4))
        for k in ("attention", "ffn", "backward"):
            out["stage_ms"][k].append(prof.get("stage_" + k, 0))
        out["attention_core_ms"].append(round(prof.get("attn_fwd", 0) + prof.get("attn_bwd", 0), 4))
        del r, dy

    def growth(v):
        return [round(b / a, 3) for a, b in zip(v, v[1:]) if a > 0]
    out["growth_per_doubling"] = {"stage_attention": growth(out["stage_ms"]["attention"]),
                                  "stage_ffn": growth(out["stage_ms"]["ffn"]),
                                  "stage_backward": growth(out["stage_ms"]["backward"]),
                                  "attention_core": growth(out["attention_core_ms"])}
    out["work_growth_per_doubling"] = {"attention_core": 4.0, "ffn": 2.0}
    return out


def _time_loop(fn, steps, warmup, stream):
    """Mean ms per call over `steps` timed calls (after `warmup`), with the
    library's per-kind events off (they sit between the kernels on the stream),
    then the per-kind spans from a second pass with them on."""
    import torch
    from megatron_transformer_layer_fwd_gb300 import mgb
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    mgb.mgb_profile_reset()
    mgb.mgb_profile_enable(True)
    n = max(1, min(steps, 5))
    for _ in range(n):
        fn()
    torch.cuda.synchronize()
    mgb.mgb_profile_enable(False)
    prof = {k: round(v[0] / n, 4) for k, v in mgb.mgb_profile_read().items() if v[1] > 0}
    if mgb.mgb_device_status(stream) != mgb.MGB_OK:
        raise RuntimeError("device error")
    return ms, prof


def _layer_line(args, name, shape, ms, prof):
    """One JSON line of --case layer / sweep: the layer's fwd+bwd time, the
    pages' three stages and the attention core, from the library's events."""
    lf = layer_flops(shape)
    gem = ("gemm_tc_fwd", "gemm_tc_dgrad", "gemm_tc_wgrad")
    return {"case": args.case, "workload": name, "dropout": args.dropout, "ms": round(ms, 4),
            "tflops": round(lf["total"] / (ms / 1e3) / 1e12, 1),
            "frac_of_nominal_2250": round(lf["total"] / (ms / 1e3) / 2.25e15, 4),
            "tokens_per_s": round(shape.tokens / (ms / 1e3), 1),
            # page 1's three segments, each between library CUDA events on the
            # stream: Attention (LN1, QKV, attention, projection + residual),
            # FFN (LN2, fc1 + activation, fc2 + residual), Backward (all of it)
            "stage_ms": {"attention": prof.get("stage_attention", 0),
                         "ffn": prof.get("stage_ffn", 0),
                         "backward": prof.get("stage_backward", 0)},
            "attention_core_ms": {"fwd": prof.get("attn_fwd", 0), "bwd": prof.get("attn_bwd", 0)},
            "gemm_ms": round(sum(prof.get(k, 0) for k in gem), 4),
            "kernel_ms": prof}


def run_case(args):
    """Sub-paths and single kernels of the step (for ncu captures and the
    sequence sweep); prints one JSON line per measurement."""
    import torch
    from megatron_transformer_layer_fwd_gb300 import build, mgb
    from megatron_transformer_layer_fwd_gb300.runner import CERunner, LayerRunner, to_device
    build.build()
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream()
    # the critical path's stream outranks the library's side streams
    hi = torch.cuda.Stream(priority=-1)
    peaks = load_peaks()
    if args.case == "gemm":
        M, N, K = args.mnk
        a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        b = torch.randn(N, K, device="cuda").to(torch.bfloat16)
        c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        d = mgb.GemmDesc(m=M, n=N, k=K, a_major=0, b_major=0, lda=K, ldb=K, ldc=N, dtype=mgb.MGB_BF16,
                         c_f32=0, accumulate=0, alpha=1.0)
        ms, prof = _time_loop(lambda: mgb.mgb_gemm(d, a, b, None, c), args.steps, args.warmup, st)
        tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
        print(json.dumps({"case": "gemm", "mnk": [M, N, K], "ms": round(ms, 4), "tflops": round(tf, 1),
                          "frac_of_burst_peak": round(tf / peaks["bf16_tflops"], 4)}))
        return
    if args.case == "gemm_f32":
        # the float32 product (forward layout) as three TF32 tensor-core
        # products, beside the FFMA path and cuBLAS float32 / single-TF32 for
        # scale; the tensor pipe runs 3 x 2MNK TF32 FLOPs, against the
        # measured bf16 burst peak x the nominal TF32 / bf16 ratio (1.1 / 2.25)
        M, N, K = args.mnk
        a = torch.randn(M, K, device="cuda")
        b = torch.randn(N, K, device="cuda")
        c = torch.empty(M, N, device="cuda")
        ws = torch.empty(mgb.mgb_gemm_f32_tc_ws_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=0, b_major=0, lda=K, ldb=K, ldc=N,
                                          dtype=mgb.MGB_F32, c_f32=0, accumulate=0, alpha=1.0),
                           epilogue=mgb.MGB_EPI_STORE, glu_block=16, ldc2=0, ldr=0, ldaux=0)
        fl = 2.0 * M * N * K
        tf32_peak = peaks["bf16_tflops"] * 1.1 / 2.25
        ref = (a.double() @ b.double().t())
        runs = [("tf32x3", lambda: mgb.mgb_gemm_f32_tc(d, a, b, None, c, ws=ws)),
                ("ffma", lambda: mgb.mgb_gemm_ex(d, a, b, None, c))]
        for name, fn in runs:
            ms, prof = _time_loop(fn, args.steps if name == "tf32x3" else 3, args.warmup, st)
            err = float(torch.linalg.norm(c.double() - ref) / torch.linalg.norm(ref))
            out = {"case": "gemm_f32_" + name, "mnk": [M, N, K], "ms": round(ms, 4),
                   "tflops": round(fl / (ms / 1e3) / 1e12, 1), "rel_l2_vs_f64": err,
                   "kernel_ms": prof}
            if name == "tf32x3":
                out["tensor_tflops"] = round(3 * fl / (ms / 1e3) / 1e12, 1)
                out["tf32_peak"] = round(tf32_peak, 1)
                out["frac_of_tf32_peak"] = round(3 * fl / (ms / 1e3) / 1e12 / tf32_peak, 4)
            print(json.dumps(out), flush=True)
        for name, tf in (("cublas_fp32", False), ("cublas_tf32_single", True)):
            torch.backends.cuda.matmul.allow_tf32 = tf
            ms, _ = _time_loop(lambda: torch.matmul(a, b.t(), out=c), 3 if not tf else args.steps,
                               args.warmup, st)
            err = float(torch.linalg.norm(c.double() - ref) / torch.linalg.norm(ref))
            print(json.dumps({"case": "gemm_f32_" + name, "mnk": [M, N, K], "ms": round(ms, 4),
                              "tflops": round(fl / (ms / 1e3) / 1e12, 1), "rel_l2_vs_f64": err}),
                  flush=True)
        torch.backends.cuda.matmul.allow_tf32 = False
        return
    if args.case == "gemm_layer":
        # the layer's twelve GEMM shapes and operand layouts (forward, input
        # gradient, weight gradient), each alone, beside torch.matmul (cuBLAS)
        # on the same operands for scale
        sh = WORKLOADS[LAYER]
        T, H, Dq = sh.tokens, sh.hidden, sh.n_q_heads * sh.head_dim
        Wqkv = (sh.n_q_heads + 2 * sh.n_kv_heads) * sh.head_dim
        F = sh.ffn
        W = 2 * F if sh.act == "swiglu" else F
        cases = [("fwd_qkv", T, Wqkv, H, 0, 0), ("fwd_proj", T, H, Dq, 0, 0), ("fwd_fc1", T, W, H, 0, 0),
                 ("fwd_fc2", T, H, F, 0, 0), ("dgrad_fc2", T, F, H, 0, 1), ("dgrad_fc1", T, H, W, 0, 1),
                 ("dgrad_proj", T, Dq, H, 0, 1), ("dgrad_qkv", T, H, Wqkv, 0, 1),
                 ("wgrad_fc2", H, F, T, 1, 1), ("wgrad_fc1", W, H, T, 1, 1), ("wgrad_proj", H, Dq, T, 1, 1),
                 ("wgrad_qkv", Wqkv, H, T, 1, 1)]
        tot_ms = tot_ref = tot_fl = 0.0
        for name, M, N, K, am, bm in cases:
            a = torch.randn(*((K, M) if am else (M, K)), device="cuda").to(torch.bfloat16)
            b = torch.randn(*((K, N) if bm else (N, K)), device="cuda").to(torch.bfloat16)
            c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
            d = mgb.GemmDesc(m=M, n=N, k=K, a_major=am, b_major=bm, lda=M if am else K,
                             ldb=N if bm else K, ldc=N, dtype=mgb.MGB_BF16, c_f32=0, accumulate=0,
                             alpha=1.0)
            ms, _ = _time_loop(lambda: mgb.mgb_gemm(d, a, b, None, c), args.steps, args.warmup, st)
            at = a.t() if am else a
            bt = b if bm else b.t()
            ref, _ = _time_loop(lambda: torch.matmul(at, bt, out=c), args.steps, args.warmup, st)
            fl = 2.0 * M * N * K
            tot_ms, tot_ref, tot_fl = tot_ms + ms, tot_ref + ref, tot_fl + fl
            print(json.dumps({"case": name, "mnk": [M, N, K], "majors": [am, bm], "ms": round(ms, 4),
                              "tflops": round(fl / ms / 1e9, 1), "cublas_ms": round(ref, 4),
                              "cublas_tflops": round(fl / ref / 1e9, 1)}), flush=True)
        print(json.dumps({"case": "gemm_layer_total", "ms": round(tot_ms, 4),
                          "tflops": round(tot_fl / tot_ms / 1e9, 1), "cublas_ms": round(tot_ref, 4),
                          "cublas_tflops": round(tot_fl / tot_ref / 1e9, 1)}), flush=True)
        return
    if args.case in ("layer", "sweep"):
        names = [LAYER] if args.case == "layer" else [f"bf16_causal_b8s{s}h2048"
                                                      for s in (128, 256, 512, 1024, 2048)]
        sweep = []
        for name in names:
            shape = WORKLOADS[name]
            r = LayerRunner(shape, layer_inputs(shape, seed=0))
            if args.dropout > 0:
                # attention-probability and hidden dropout at the same rate, the
                # sites' states drawn from the tensor-parallel RNG tracker
                r.desc.attn_dropout = r.desc.hidden_dropout = args.dropout
                mgb.mgb_block_dropout_plan(r.desc, mgb.rng_tracker(1234))
                saved, _, bwd = mgb.mgb_block_sizes(r.desc)
                r.saved = torch.empty(saved, dtype=torch.uint8, device="cuda")
                r.ws = torch.empty(bwd, dtype=torch.uint8, device="cuda")
            dy = torch.full_like(r.x, 1.0 / (shape.tokens * shape.hidden))
            variants = [("high-priority stream, side streams", hi, "1")]
            if args.case == "layer":
                variants += [("default-priority stream, side streams", st, "1"),
                             ("high-priority stream, serial (MGB_SIDE_STREAMS=0)", hi, "0")]
            for vname, vst, side in variants:
                os.environ["MGB_SIDE_STREAMS"] = side

                def fb():
                    r.fwd(vst)
                    r.bwd(dy, vst)
                ms, prof = _time_loop(fb, args.steps, args.warmup, vst)
                os.environ.pop("MGB_SIDE_STREAMS", None)
                out = _layer_line(args, name, shape, ms, prof)
                out["streams"] = vname
                if args.case == "sweep":
                    sweep.append((shape.seq, out["stage_ms"], out["attention_core_ms"]))
                print(json.dumps(out), flush=True)
            del r
        if args.case == "sweep":
            # growth per doubling of seq: attention work grows 4x (S^2), the
            # FFN's 2x (linear in tokens) at fixed batch
            def growth(f):
                return [round(f(b) / f(a), 3) for a, b in zip(sweep, sweep[1:]) if f(a) > 0]
            print(json.dumps({
                "case": "sweep_summary", "seq": [q for q, _, _ in sweep],
                "stage_ms": {k: [st_[k] for _, st_, _ in sweep] for k in ("attention", "ffn", "backward")},
                "growth_per_doubling": {
                    "stage_attention": growth(lambda e: e[1]["attention"]),
                    "stage_ffn": growth(lambda e: e[1]["ffn"]),
                    "stage_backward": growth(lambda e: e[1]["backward"]),
                    "attention_core_fwd_bwd": growth(lambda e: e[2]["fwd"] + e[2]["bwd"])},
                "work_growth": {"attention_core": 4.0, "ffn": 2.0}}), flush=True)
        return
    if args.case == "attention":
        # the attention core of the layer workload: forward, then backward
        # (q, k, v as column slices of one fused buffer, as in the layer)
        shape = WORKLOADS[LAYER]
        B, S, nq, nkv, d = shape.batch, shape.seq, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
        W = (nq + 2 * nkv) * d
        g = torch.Generator(device="cuda").manual_seed(0)
        qkv = torch.randn((B * S, W), device="cuda", generator=g).to(torch.bfloat16)
        o = torch.empty((B * S, nq * d), device="cuda", dtype=torch.bfloat16)
        lse = torch.empty((B, nq, S), device="cuda")
        dout = torch.randn((B * S, nq * d), device="cuda", generator=g).to(torch.bfloat16)
        dqkv = torch.empty_like(qkv)
        ws = torch.empty(mgb.mgb_attention_bwd_ws_bytes(B, S, nq), dtype=torch.uint8, device="cuda")
        cz = int(shape.causal)
        q, k, v = qkv, qkv[:, nq * d:], qkv[:, (nq + nkv) * d:]

        def fwd():
            mgb.mgb_attention_fwd(B, S, nq, nkv, d, cz, mgb.MGB_BF16, q, k, v, W, W, o, lse)

        def bwd():
            mgb.mgb_attention_bwd(B, S, nq, nkv, d, cz, mgb.MGB_BF16, q, k, v, W, W, o, lse, dout,
                                  nq * d, dqkv, dqkv[:, nq * d:], dqkv[:, (nq + nkv) * d:], W, W, ws)
        # FLOPs: forward 2 products (S, PV); backward 5 (S, dP, dV, dK, dQ) = 2.5x
        fl = layer_flops(shape)["attn_fwd"]
        for name, fn, f in (("attention_fwd", fwd, fl), ("attention_bwd", bwd, 2.5 * fl)):
            ms, prof = _time_loop(fn, args.steps, args.warmup, st)
            print(json.dumps({"case": name, "workload": LAYER, "ms": round(ms, 4),
                              "tflop": round(f / 1e12, 4), "tflops": round(f / (ms / 1e3) / 1e12, 1),
                              "kernel_ms": prof}), flush=True)
        return
    if args.case == "ln":
        # the layer's LayerNorms at its shape (T 8192, H 4096, bf16, affine):
        # forward (the warp-per-row kernel, and the block-per-row kernel for
        # comparison) and backward with the residual input (plus its
        # dgamma/dbeta partial-sum reduction)
        T, H = WORKLOADS[LAYER].tokens, WORKLOADS[LAYER].hidden
        g = torch.Generator(device="cuda").manual_seed(0)
        mk = lambda *sh: torch.randn(*sh, device="cuda", generator=g).to(torch.bfloat16)
        x, dy, dres, gm, bt = mk(T, H), mk(T, H), mk(T, H), mk(H), mk(H)
        y, dx = torch.empty_like(x), torch.empty_like(x)
        mu = torch.empty(T, device="cuda")
        rs = torch.empty(T, device="cuda")
        dg, db = torch.empty_like(gm), torch.empty_like(bt)
        ws = torch.empty(mgb.mgb_layernorm_bwd_ws_bytes(T, H), dtype=torch.uint8, device="cuda")
        fwd_bytes = 2 * T * H * 2 + 8 * T
        bwd_bytes = 4 * T * H * 2 + 8 * T
        fwd = lambda: mgb.mgb_layernorm_fwd(T, H, mgb.MGB_BF16, 1e-5, x, gm, bt, y, mu, rs, hi)
        bwd = lambda: mgb.mgb_layernorm_bwd(T, H, mgb.MGB_BF16, x, mu, rs, gm, dy, dres, dx, dg, db,
                                            ws, hi)
        # MGB_LN_KERNEL: tma (rows streamed into shared memory by bulk copies;
        # the forward's default), warp (register prefetch, forward only), block
        # (block per row; backward: register prefetch), async (backward's
        # default: per-thread asynchronous copies into a shared-memory ring)
        for name, env, fn, nb in (("layernorm_fwd_tma", "tma", fwd, fwd_bytes),
                                  ("layernorm_fwd_warp", "warp", fwd, fwd_bytes),
                                  ("layernorm_fwd_block", "block", fwd, fwd_bytes),
                                  ("layernorm_bwd_async", "async", bwd, bwd_bytes),
                                  ("layernorm_bwd_tma", "tma", bwd, bwd_bytes),
                                  ("layernorm_bwd_block", "block", bwd, bwd_bytes)):
            os.environ["MGB_LN_KERNEL"] = env
            ms, prof = _time_loop(fn, args.steps, args.warmup, hi)
            os.environ.pop("MGB_LN_KERNEL", None)
            gbs = nb / (ms / 1e3) / 1e9
            print(json.dumps({"case": name, "tokens": T, "hidden": H, "ms": round(ms, 4),
                              "algorithmic_bytes": nb, "gbs": round(gbs, 1),
                              "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "kernel_ms": prof}),
                  flush=True)
        return
    if args.case == "embedding":
        # the input-side lookup of the tied table (vocab-parallel embedding, one
        # shard = the whole vocabulary) at the CE workload's sizes; ids drawn
        # like the CE targets (uniform); backward accumulated onto the table's
        # gradient (the tied form)
        ce = CE_WORKLOADS[CE]
        T, H, V = ce.tokens, ce.hidden, ce.vocab
        g = torch.Generator(device="cuda").manual_seed(0)
        ids = torch.randint(0, V, (T,), device="cuda", generator=g, dtype=torch.int32)
        E = torch.randn((V, H), device="cuda", generator=g).to(torch.bfloat16)
        out = torch.empty((T, H), device="cuda", dtype=torch.bfloat16)
        dout = torch.randn((T, H), device="cuda", generator=g).to(torch.bfloat16)
        dE = torch.zeros((V, H), device="cuda", dtype=torch.bfloat16)
        ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(T, 0, V), dtype=torch.uint8, device="cuda")
        uniq = int(torch.unique(ids).numel())
        ws2 = torch.empty_like(ws)
        plan = mgb.mgb_embedding_bwd_prepare(T, 0, V, ids, ws2)
        fwd_bytes = 2 * T * H * 2                         # rows read + out written
        bwd_bytes = T * H * 2 + 2 * uniq * H * 2 + 16 * T  # dout, touched rows in/out, ids+lists
        for name, fn, nb in (
                ("embedding_fwd", lambda: mgb.mgb_embedding_fwd(T, H, 0, V, mgb.MGB_BF16, ids, E, out),
                 fwd_bytes),
                ("embedding_bwd_accumulate",
                 lambda: mgb.mgb_embedding_bwd(T, H, 0, V, mgb.MGB_BF16, ids, dout, dE, 1, ws), bwd_bytes),
                # the same backward in two steps: the token order from the ids
                # alone (index work, no HBM-bound part), then the row sums
                ("embedding_bwd_prepare",
                 lambda: mgb.mgb_embedding_bwd_prepare(T, 0, V, ids, ws2), 0),
                ("embedding_bwd_apply_accumulate",
                 lambda: mgb.mgb_embedding_bwd_apply(plan, H, mgb.MGB_BF16, dout, dE, 1), bwd_bytes)):
            ms, prof = _time_loop(fn, args.steps, args.warmup, st)
            line = {"case": name, "tokens": T, "hidden": H, "vocab": V, "unique_ids": uniq,
                    "ms": round(ms, 4), "kernel_ms": prof}
            if nb:
                gbs = nb / (ms / 1e3) / 1e9
                line.update({"algorithmic_bytes": nb, "gbs": round(gbs, 1),
                             "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)})
            print(json.dumps(line), flush=True)
        return
    if args.case == "ce":
        ce = CE_WORKLOADS[CE]
        if args.ce_shape:
            # a smaller case of the same kernels (for counter captures)
            T_, H_, V_, C_ = (int(v) for v in args.ce_shape.split(","))
            ce = CEShape(T_, H_, V_, C_)
        cin = ce_inputs(ce, seed=0)
        hid = to_device(cin["hidden"], torch.bfloat16)
        emb = to_device(cin["emb"], torch.bfloat16)
        tg = torch.from_numpy(cin["targets"]).to("cuda")
        cf = ce_flops(ce)
        modes = [(mgb.MGB_CE_STREAM, "stream", 0), (mgb.MGB_CE_FUSED, "fused", 0),
                 (mgb.MGB_CE_RESIDENT, "resident", 0), (mgb.MGB_CE_BLOCKED, "blocked",
                                                        args.token_block)]
        if args.ce_mode == "blocked" and args.token_block == 0:
            modes += [(mgb.MGB_CE_BLOCKED, "blocked", tb) for tb in (1024, 4096)]
        modes = [m for m in modes if args.ce_mode in (m[1], "all")]
        for mode, name, tb in modes:
            r = CERunner(ce.tokens, ce.hidden, ce.vocab, ce.chunk, hid, emb, tg, mode=mode,
                         token_block=tb)
            ms, prof = _time_loop(lambda: r.run(hi), args.steps, args.warmup, hi)
            out = {"case": "ce", "mode": name, "ms": round(ms, 4),
                   "tflops": round(cf["total"] / (ms / 1e3) / 1e12, 1),
                   "workspace_gb": round(r.ws.numel() / 1e9, 3), "kernel_ms": prof}
            if mode == mgb.MGB_CE_BLOCKED:
                out["token_block"] = r.token_block
            if mode in (mgb.MGB_CE_STREAM, mgb.MGB_CE_FUSED):
                out["tflops_with_recompute"] = round((cf["total"] + cf["recompute"]) / (ms / 1e3) / 1e12, 1)
            if mode == mgb.MGB_CE_STREAM:
                sb = ce_stream_bytes(ce)
                sms = prof.get("ce_stats", 0) + prof.get("ce_grad", 0)
                out.update({"stream_ms": round(sms, 4), "stream_gbs": round(sb / (sms / 1e3) / 1e9, 1),
                            "frac_of_hbm": round(sb / (sms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)})
            print(json.dumps(out), flush=True)
            del r
        return
    raise SystemExit(f"unknown case {args.case}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sequence sweep of the causal workloads in the step run")
    ap.add_argument("--case", default="step",
                    choices=("step", "layer", "sweep", "ce", "gemm", "gemm_f32", "gemm_layer",
                             "attention", "embedding", "ln"),
                    help="step (default: the whole hot path, one JSON line) or a sub-path / single kernel")
    ap.add_argument("--mnk", type=int, nargs=3, default=(8192, 22016, 4096))
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="--case layer|sweep: attention and hidden dropout probability")
    ap.add_argument("--ce-mode", default="all",
                    choices=("all", "stream", "fused", "resident", "blocked"),
                    help="--case ce: which CE mode(s) to time")
    ap.add_argument("--ce-shape", default="",
                    help="--case ce: tokens,hidden,vocab,chunk instead of the CE workload's")
    ap.add_argument("--token-block", type=int, default=0,
                    help="tokens per block of the blocked CE (0: the library's default)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case != "step":
        run_case(args)
        return
    world, rank, local = dist_setup()

    if args.impl == "reference":
        # the reference arm is the float64 oracle on the host cores, rank 0 only
        if rank != 0:
            return
        sample = OracleSample()
        for _ in range(args.warmup):
            sample.run_once()
        secs = statistics.median(sample.run_once() for _ in range(args.steps))
        tfl = sample.flops / secs / 1e12
        per_step = [{"sample": f"1 x [{sample.desc}] per step"}]
        out = {"impl": "reference", "metric": METRIC, "value": round(tfl, 6), "unit": "TFLOP/s",
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(secs * 1e3, 1), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f64", "data": "synthetic",
               "config": {"workload": WORKLOAD, "parallelism": "host cores, rank 0 only"},
               "cpu_baseline": {"value": round(tfl, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": per_step[0]["sample"]},
               "e2e": {"value": round(tfl, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(out), flush=True)
        return

    # CPU baseline first (before any CUDA context: no fork after GPU use here)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = OracleSample().timed(budget_s=12.0)
    out = run_ours(args, world, rank, local)
    if rank == 0:
        if cpu is not None:
            out["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
