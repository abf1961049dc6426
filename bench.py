#!/usr/bin/env python
"""Benchmark of one DFlash draft step + greedy verify on GB300.

A step = dflash_ctx_fuse (new context rows) + dflash_draft_block (K/V append
in the same weight pass, non-causal block pass, LM head + argmax) +
dflash_synth_target (stand-in for the target's verify tokens, agreement
probability p per position) + dflash_verify_greedy, for the whole batch,
captured once in a CUDA graph and replayed.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (bounded sample of the same workload).
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workload as W  # noqa: E402

METRIC = ("draft block tokens/s & accepted tokens/s at block 16, 1 GB300; "
          "% HBM/tensor roofline")
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_8b_b1", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--accept-sample", type=int, default=200)
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3"],
                    help="drafter context cache: bf16, or E4M3 codes with per-vector scales")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ------------------------------------------------------------ accounting
def step_bytes(wl, ctx_before, new_rows, kv="bf16"):
    """Algorithmic HBM bytes of one step: every weight once, the context K/V
    read once per layer, the appended K/V written once, the step's inputs and
    outputs.  An E4M3 cache holds one byte per element and a 4-byte scale
    per (position, head) vector."""
    d = wl.draft
    H, kvd = d.hidden, d.kv_dim
    weights = (H * d.n_taps * H + H) + d.n_layers * d.layer_params() + H + H \
        + d.vocab * H + d.n_layers * H * d.conv_width
    L_after = np.asarray(ctx_before) + np.asarray(new_rows)
    kv_elems = (int(L_after.sum()) + int(np.sum(new_rows))) * 2 * kvd * d.n_layers
    kv_b = 2.0 if kv == "bf16" else 1.0 + 4.0 / d.head_dim
    taps = int(np.sum(new_rows)) * d.n_taps * H
    emb = wl.batch * H
    return int(2 * (weights + taps + emb) + kv_b * kv_elems)


def step_flops(wl, ctx_before, new_rows):
    d = wl.draft
    rows = wl.batch * d.block
    T = int(np.sum(new_rows))
    H = d.hidden
    dense = 2 * T * H * d.n_taps * H
    dense += d.n_layers * (2 * (rows + T) * d.qkv_rows * H + 2 * rows * H * d.q_dim
                           + 2 * rows * 3 * d.mlp * H)
    dense += 2 * rows * d.vocab * H
    keys = np.asarray(ctx_before) + np.asarray(new_rows) + d.block
    attn = d.n_layers * 4 * d.block * d.n_q_heads * d.head_dim * int(keys.sum())
    return dense + attn


def phase_roofline(wl, ctx_before, new_rows, kv, hbm_gbs, tc_tflops):
    """Lower bound on the step time as a sum over its two kinds of phase,
    each at max(bytes / HBM bandwidth, flops / tensor rate): attention
    (context K/V read once per layer, QK^T and PV flops) and the GEMMs
    (every other algorithmic byte, the dense flops).  Equals the HBM-only
    bound when both phases are bandwidth-bound (batch 1, DFlash-2); larger
    when the GEMMs are tensor-bound (batch 32)."""
    d = wl.draft
    kv_b = 2.0 if kv == "bf16" else 1.0 + 4.0 / d.head_dim
    L_after = np.asarray(ctx_before) + np.asarray(new_rows)
    attn_bytes = kv_b * int(L_after.sum()) * 2 * d.kv_dim * d.n_layers
    keys = np.asarray(ctx_before) + np.asarray(new_rows) + d.block
    attn_flops = d.n_layers * 4 * d.block * d.n_q_heads * d.head_dim * int(keys.sum())
    total_bytes = step_bytes(wl, ctx_before, new_rows, kv)
    gemm_bytes = total_bytes - attn_bytes
    gemm_flops = step_flops(wl, ctx_before, new_rows) - attn_flops
    t_attn = max(attn_bytes / (hbm_gbs * 1e9), attn_flops / (tc_tflops * 1e12))
    t_gemm = max(gemm_bytes / (hbm_gbs * 1e9), gemm_flops / (tc_tflops * 1e12))
    return {"t_min_ms": (t_attn + t_gemm) * 1e3, "attention_ms": t_attn * 1e3, "gemm_ms": t_gemm * 1e3,
            "gemm_bound": "tensor" if gemm_flops / (tc_tflops * 1e12) > gemm_bytes / (hbm_gbs * 1e9)
            else "hbm"}


def acceptance_profile(hist, p):
    """Per-position acceptance from hist[n] = number of (request, step)
    samples that accepted n drafts (n = 0..B-1).  Block position i (1-based)
    is accepted when n >= i.  The synthetic target agrees with the draft at
    each position independently with its request's probability p_b, so the
    expected rate at position i is the mean over requests of p_b**i."""
    hist = np.asarray(hist, dtype=np.float64)
    total = float(hist.sum())
    n = np.arange(hist.size)
    at_least = np.cumsum(hist[::-1])[::-1][1:] / total  # P(n >= i), i = 1..B-1
    expected = np.mean(np.asarray(p, dtype=np.float64)[:, None] ** n[None, 1:], axis=0)
    return {"samples": int(total),
            "mean_accepted_drafts": float((hist * n).sum() / total),
            "p_accept_at_position": [round(float(x), 4) for x in at_least],
            "expected_p_accept_at_position": [round(float(x), 4) for x in expected]}


def lm_head_bytes(d, rows):
    return 2 * d.vocab * d.hidden + 2 * rows * d.hidden + 4 * rows


def source_sha():
    """Hash of the sources the LM-head GEMM kernel is compiled from."""
    h = hashlib.sha256()
    for f in ("gemm_tc05.cu", "epilogue.cuh", "common.cuh", "kernels.h"):
        h.update(open(os.path.join(ROOT, "block_diffusion_speculative_fuse_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(config):
    """DRAM bytes per LM-head launch from the committed ncu summary, or None
    when the summary is missing or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", f"lm_head_gemm_{config}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"source_sha:\s*([0-9a-f]+)", txt)
    if not m or not s or s.group(1) != source_sha():
        return None
    return float(m.group(1))


# ------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.dev = dev_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"unavailable": "nvidia-smi not runnable"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"unavailable": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ oracle timing
def oracle_step_fn(wl, host):
    """The oracle's version of one step on the same inputs (no tuning)."""
    import oracle as O
    d = wl.draft
    dws = O.LayerStack(d, host["weights"], host["shared"])
    taps = O.bf16_to_f64(host["taps"])
    ctx_before = W.ctx_lengths(wl)
    new_rows = W.new_row_counts(wl)
    ks0 = {k: O.bf16_to_f64(v) for k, v in host["ctx_k"].items()}
    vs0 = {k: O.bf16_to_f64(v) for k, v in host["ctx_v"].items()}

    def run():
        c = O.ctx_fuse(d, dws, taps)
        o = 0
        drafts = []
        for r in range(wl.batch):
            C, T = int(ctx_before[r]), int(new_rows[r])
            ks, vs = [], []
            for l in range(d.n_layers):
                kn, vn = O.ctx_kv(d, dws, l, c[o:o + T], np.arange(C, C + T))
                ks.append(np.concatenate([ks0[(l, r)], kn]) if C else kn)
                vs.append(np.concatenate([vs0[(l, r)], vn]) if C else vn)
            o += T
            dr, _ = O.draft_block(d, dws, int(host["anchor"][r]), C + T, ks, vs)
            drafts.append(dr)
        drafts = np.array(drafts)
        t = W.synth_target_ids(drafts, W.agreement_probs(wl), d.vocab, 1, 0)
        return O.verify_batch(drafts, t, ctx_before + new_rows, ctx_before + new_rows)
    return run


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(wl, host, n_steps, n_warm):
    run = oracle_step_fn(wl, host)
    for _ in range(n_warm):
        run()
    t0 = time.perf_counter()
    for _ in range(n_steps):
        run()
    return (time.perf_counter() - t0) / max(1, n_steps)


def host_inputs_for_oracle(wl):
    d = wl.draft
    wid = wl.wid
    ctx_before = W.ctx_lengths(wl)
    new_rows = W.new_row_counts(wl)
    host = {"weights": W.draft_weights(d, wid), "shared": W.shared_weights(d, wid),
            "taps": W.taps_bf16(int(new_rows.sum()), d, wid),
            "anchor": W.uniform_tokens(wl.batch, d.vocab, wid, W.TENSOR_IDS["anchor"]),
            "ctx_k": {}, "ctx_v": {}}
    for l in range(d.n_layers):
        for r in range(wl.batch):
            n = int(ctx_before[r])
            if n:
                host["ctx_k"][(l, r)] = W.context_kv_bf16(d, wid, l, r, n, "k")
                host["ctx_v"][(l, r)] = W.context_kv_bf16(d, wid, l, r, n, "v")
    return host


# ------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = W.get_workload(args.config)
    host = host_inputs_for_oracle(wl)
    sec = time_oracle(wl, host, args.steps, args.warmup)
    d = wl.draft
    value = wl.batch * (d.block - 1) / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "block": d.block},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"full oracle draft step of {wl.name} per step "
                                   f"(fuse, K/V append, block draft, verify)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ our arm
def e4m3_vs_bf16(st, wl, stream):
    """The draft of one step with the E4M3 context cache against the same
    step (same weights, inputs and context) over a bf16 cache: the fraction
    of drafted tokens that agree, and the mean length of the matching prefix
    of each request's block, which is the number of drafts an E4M3 drafter
    gets accepted by a target that accepts exactly the bf16 drafter's block.
    With random-init weights the logits are nearly flat, so this understates
    the agreement of a trained drafter."""
    import torch

    from block_diffusion_speculative_fuse_gb300.session import DraftStep
    st16 = DraftStep(wl, model=st.model)
    with torch.cuda.stream(stream):
        st.fuse(stream)
        st.draft_block(stream=stream, append=True)
        st16.fuse(stream)
        st16.draft_block(stream=stream, append=True)
    stream.synchronize()
    a, b = st.draft.cpu().numpy(), st16.draft.cpu().numpy()
    same = a == b
    prefix = np.where(same.all(1), same.shape[1], np.argmin(same, axis=1))
    del st16
    return {"drafted_token_agreement": float(same.mean()),
            "mean_matching_prefix": float(prefix.mean()), "block_drafts": int(same.shape[1]),
            "requests": int(same.shape[0])}


def run_ours(args, rank, world, dist):
    import torch

    from block_diffusion_speculative_fuse_gb300 import _build, binding as B
    from block_diffusion_speculative_fuse_gb300.session import DraftStep

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _build.build()
    B.load()
    wl = W.get_workload(args.config)
    d = wl.draft
    st = DraftStep(wl, kv_dtype=args.kv)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    # launches per step, counted on one eager step
    with torch.cuda.stream(stream):
        n0 = B.dflash_kernel_launches()
        st.step(stream)
        launches_per_step = B.dflash_kernel_launches() - n0
    stream.synchronize()
    status = st.status()
    if status[0] != 0:
        raise RuntimeError(f"device status {status} after the first step")

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            st.step(stream)
        torch.cuda.synchronize()

    def one():
        if graph is not None:
            graph.replay()
        else:
            st.step(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one()
    stream.synchronize()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            one()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, dist)
    clocks = sampler.stop() if rank == 0 else None

    status = st.status()
    if status[0] != 0:
        raise RuntimeError(f"device status {status} after the timed steps")

    # acceptance: mean emitted tokens per step over fresh synthetic draws, and
    # the histogram of accepted draft counts (per-position acceptance)
    acc = torch.zeros(wl.batch, dtype=torch.int64, device="cuda")
    hist = torch.zeros(d.block, dtype=torch.int64, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(args.accept_sample):
            one()
            acc += st.n_accept.long() + 1
            hist += torch.bincount(st.n_accept.long(), minlength=d.block)[:d.block]
    stream.synchronize()
    emitted_per_step = float(acc.sum().item()) / args.accept_sample
    accept_profile = acceptance_profile(hist.cpu().numpy(), W.agreement_probs(wl))

    # e2e through host buffers: H2D of the step's inputs, D2H of its outputs
    pin = lambda t: t.cpu().pin_memory()
    h_in = [(pin(st.taps), st.taps), (pin(st.anchor), st.anchor),
            (pin(st.anchor_pos), st.anchor_pos), (pin(st.pending_req), st.pending_req),
            (pin(st.pending_pos), st.pending_pos)]
    h_out = [(st.out_tokens, torch.empty_like(st.out_tokens, device="cpu").pin_memory()),
             (st.n_accept, torch.empty_like(st.n_accept, device="cpu").pin_memory()),
             (st.draft, torch.empty_like(st.draft, device="cpu").pin_memory())]
    h2d = sum(h.numel() * h.element_size() for h, _ in h_in)
    d2h = sum(h.numel() * h.element_size() for _, h in h_out)
    ke = max(10, args.steps // 2)
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e2.record(stream)
        for _ in range(ke):
            for h, dv in h_in:
                dv.copy_(h, non_blocking=True)
            one()
            for dv, h in h_out:
                h.copy_(dv, non_blocking=True)
        e3.record(stream)
    e3.synchronize()
    ms_e2e = max_over_ranks(e2.elapsed_time(e3) / ke, dist)

    # dominant kernel: the LM-head GEMM (+ its argmax reduce), timed alone
    rows = wl.batch * d.block
    x = torch.randn((rows, d.hidden), device="cuda").to(torch.bfloat16)
    am = torch.zeros(rows, dtype=torch.int32, device="cuda")
    nl = max(20, args.steps // 4)
    with torch.cuda.stream(stream):
        for _ in range(5):
            B.dflash_lm_head_argmax(st.model.handle, x, rows, am, None, st.ws, stream)
        e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e4.record(stream)
        for _ in range(nl):
            B.dflash_lm_head_argmax(st.model.handle, x, rows, am, None, st.ws, stream)
        e5.record(stream)
    e5.synchronize()
    ms_lm = e4.elapsed_time(e5) / nl

    kv_cmp = None
    if args.kv == "e4m3":
        kv_cmp = e4m3_vs_bf16(st, wl, stream)

    if rank != 0:
        return
    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    sb = step_bytes(wl, st.ctx_before, st.new_rows, args.kv)
    # a step's kernels run back to back for a long time: the sustained rate
    tc = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops", 1700.0)))
    phase = phase_roofline(wl, st.ctx_before, st.new_rows, args.kv, hbm, tc)
    sf = step_flops(wl, st.ctx_before, st.new_rows)
    steps_per_s = 1e3 / ms
    drafted = whole_job_rate(wl.batch * (d.block - 1), ms, world)
    accepted = whole_job_rate(emitted_per_step, ms, world)
    lmb = lm_head_bytes(d, rows)
    lm_gbs = lmb / (ms_lm * 1e-3) / 1e9
    traffic = profiled_traffic(wl.name)
    step_gbs = sb / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": drafted, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random-init weights, random taps and context K/V)",
        "config": {"workload": wl.name, "batch": wl.batch, "block": d.block,
                   "ctx_len": int(st.ctx_before.max()), "new_ctx_rows": int(st.T),
                   "draft_layers": d.n_layers, "hidden": d.hidden, "vocab": d.vocab,
                   "kv_cache": args.kv, "cuda_graph": graph is not None,
                   "l2": "inputs larger than L2: %.2f GB streamed per step" % (sb / 1e9)},
        "steps_per_s": steps_per_s,
        "drafted_tokens_per_s": drafted,
        "accepted_tokens_per_s": accepted,
        "emitted_tokens_per_step": emitted_per_step,
        "acceptance": accept_profile,
        "step_roofline": {"bound": "hbm", "bytes": sb, "flops": sf, "achieved": step_gbs,
                          "peak": hbm, "unit": "GB/s", "frac": step_gbs / hbm,
                          "peak_kind": pk_kind},
        "phase_roofline": dict(phase, frac=phase["t_min_ms"] / ms, tensor_peak_tflops=tc,
                               bound="mixed" if phase["gemm_bound"] == "tensor" else "hbm"),
        "roofline": {"bound": "hbm", "kernel": "gemm_tc05 LM head + argmax (151936x4096)",
                     "achieved": lm_gbs, "peak": hbm, "unit": "GB/s", "frac": lm_gbs / hbm,
                     "traffic": traffic, "bytes_per_launch": lmb, "ms_per_launch": ms_lm,
                     "peak_kind": pk_kind},
        "e2e": {"value": whole_job_rate(wl.batch * (d.block - 1), ms_e2e, world),
                "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_e2e},
        "gpu_launches": int(launches_per_step * args.steps),
        "launches_per_step": int(launches_per_step),
        "clocks": clocks,
    }
    if kv_cmp is not None:
        line["kv_e4m3_vs_bf16"] = kv_cmp
    if world == 1 and not args.no_cpu_baseline:
        host = host_inputs_for_oracle(wl)
        sec = time_oracle(wl, host, 1, 0)
        line["cpu_baseline"] = {
            "value": wl.batch * (d.block - 1) / sec, "unit": "tokens/s", "cores": cores(),
            "kind": "oracle",
            "sample": f"one full oracle step of {wl.name} (fp64 NumPy: fuse, K/V append, "
                      f"block draft, LM head, verify), {sec:.2f} s"}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ end-to-end loop
def run_e2e(args, rank, world):
    """Greedy speculative decoding with a target model (tiny_e2e, e2e_8layer):
    accepted tokens/s, the draft share of the decode time and token identity
    against the same target's autoregressive greedy output (GPU)."""
    import torch

    from block_diffusion_speculative_fuse_gb300 import _build, binding as B
    from block_diffusion_speculative_fuse_gb300.device import DeviceModel, i32
    from block_diffusion_speculative_fuse_gb300.generate import SpecDecoder, TargetRunner, \
        ar_generate

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    _build.build()
    B.load()
    wl = W.get_workload(args.config)
    ts, ds = wl.target, wl.draft
    shared = W.shared_weights(ts, wl.wid)
    tm = DeviceModel(ts, W.target_weights(ts, wl.wid), shared, draft=False)
    dm = DeviceModel(ds, W.draft_weights(ds, wl.wid), {k: tm.t[k] for k in ("embed", "lm_head")},
                     draft=True)
    b, P, N = wl.batch, wl.prompt_len, wl.gen_tokens
    prompts = W.uniform_tokens(b * P, ts.vocab, wl.wid, W.TENSOR_IDS["prompt"]).reshape(b, P)
    # draft vs target time inside the speculative loop: CUDA event pairs
    # around each call, read after the loop (no synchronisation inside it)
    ev = {"draft": [], "target": []}
    orig_db, orig_tf = B.dflash_draft_block, B.dflash_target_forward

    def timed(name, fn):
        def w(*a, **k):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            r = fn(*a, **k)
            e1.record()
            ev[name].append((e0, e1))
            return r
        return w

    sd = SpecDecoder(tm, dm, wl.tap_layers, b, P + N)
    sd.generate(prompts[:, :min(P, 32)], 8)  # warm-up (kernels, workspaces)
    sd = SpecDecoder(tm, dm, wl.tap_layers, b, P + N)
    B.dflash_draft_block = timed("draft", orig_db)
    B.dflash_target_forward = timed("target", orig_tf)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        spec = sd.generate(prompts, N)
        torch.cuda.synchronize()
        t_spec = time.perf_counter() - t0
    finally:
        B.dflash_draft_block, B.dflash_target_forward = orig_db, orig_tf
    torch.cuda.synchronize()
    ev = {k: sum(a.elapsed_time(b_) for a, b_ in v) for k, v in ev.items()}
    runner = TargetRunner(tm, b, P + N + 1, P)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ar = ar_generate(runner, prompts, N)
    torch.cuda.synchronize()
    t_ar = time.perf_counter() - t0
    n_iter = len(sd.stats) // b
    line = {
        "metric": "accepted tokens/s (greedy speculative decoding, end to end)",
        "value": b * N / t_spec, "unit": "tokens/s", "n_gpus": world, "steps": n_iter,
        "warmup": 1, "ms_per_step": t_spec * 1e3 / max(1, n_iter), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random-init target and drafter, uniform prompts)",
        "config": {"workload": wl.name, "batch": b, "prompt": P, "generate": N,
                   "block": ds.block, "target_layers": ts.n_layers,
                   "draft_layers": ds.n_layers},
        "token_identical_to_ar": bool(np.array_equal(spec, ar)),
        "mean_accepted_per_iteration": float(np.mean(sd.stats)) if sd.stats else 0.0,
        "draft_ms_total": ev["draft"], "target_ms_total": ev["target"],
        "draft_share_of_loop": ev["draft"] / (t_spec * 1e3),
        "ar_tokens_per_s": b * N / t_ar,
        "note": "wall clock includes the prefill; the loop state stays on the device and each "
                "iteration reads back the emitted counts (batch int32) for the stop test",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------ ranks
def check_world(gpus, world):
    """--gpus must name the number of ranks the launcher started (one per
    GPU); N > 1 is launched through torch.distributed.run."""
    if gpus != world:
        raise SystemExit(f"--gpus {gpus} but {world} rank(s) were launched: run "
                         f"`python -m torch.distributed.run --nproc-per-node {gpus} bench.py "
                         f"--gpus {gpus} ...` (or omit --gpus for one GPU)")


def max_over_ranks(x, dist):
    """The largest value of x over all ranks (the job's time is its slowest
    rank's): an all-reduce on the GPU under NCCL, on the host under gloo."""
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, ms_max, world):
    """Units per second of the whole job: every rank processes the same
    per-step work (weak scaling), timed by the slowest rank's step."""
    return units_per_rank_step * world * 1e3 / ms_max


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    check_world(args.gpus, world)
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group(backend=backend)
        dist = tdist
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif W.get_workload(args.config).target is not None:
        if args.kv != "bf16":
            raise SystemExit("--kv e4m3 applies to the draft-step workloads only")
        run_e2e(args, rank, world)
    else:
        run_ours(args, rank, world, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
