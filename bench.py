#!/usr/bin/env python3
"""Throughput of exact attention (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5] [--impl ours|reference]

One step is the whole hot path on one batch of synthetic input: the forward
kernel (O and lse), then the backward's two kernels: dQ (which also forms
each row's D = rowsum(dO * O) and lse in base 2) and dK / dV.  The
default workload is the training configuration B=8, H=16, N=4096, d=128,
causal, forward + backward.  Inputs (seeded bf16 draws) are resident in HBM
before timing; they total 537 MB, larger than the 129 MB L2, so no L2 flush
is inserted between steps.  Workloads whose inputs are below twice the L2
write a 258 MB buffer before every timed step instead, and their step time
is then the sum of the per-step CUDA-event durations (flush excluded).

Work convention: forward 4*B*H*N^2*d (halved when causal), backward 2.5x the
forward.  ``value`` = total TFLOP/s of the timed steps (all ranks).

Extra keys on the JSON line:
  roofline      the dominant kernel's achieved rate (CUDA events on its own
                stream, averaged over the timed steps) against the measured
                peak in MEASURED_PEAKS.json, plus its DRAM traffic per launch
                from the committed ncu summary (null if the kernel changed)
  cpu_baseline  the fp64 CPU oracle timed on this host on a bounded sample
  e2e           the same metric through the C ABI with pinned HOST buffers:
                host->device copies of Q, K, V, dO and device->host copies of
                O, lse, dQ, dK, dV inside the timed region, every step,
                pipelined with the compute (two buffer slots, two copy
                streams)
  clocks        nvidia-smi samples taken during the timed region
``--impl reference`` times the CPU oracle (the only other implementation of
this path) on the same workload, one bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (bf16, 1×GB300) and % of dense BF16 tensor peak"
UNIT = "TFLOPS"
L2_BYTES = 129_000_000
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="c5")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def workload_desc(w):
    if w.kind == "masked":
        what = (f"sliding window (left {w.window[0]}, right {w.window[1]})" if w.window is not None
                else f"prefix-LM boolean mask (prefix {w.prefix})" if w.prefix is not None
                else f"additive {'bf16' if w.bias_bf16 else 'float32'} mask -{w.bias_slope:g}*|i-j| shared by all heads")
        return (f"{w.name}: B={w.B} H={w.H} Hkv={w.Hkv} N={w.N} d={w.d} {'causal ' if w.causal else ''}{what} "
                f"{'fwd+bwd' if w.with_grad else 'fwd'}; FLOPs count the visible (query, key) pairs")
    if w.kind == "varlen":
        from sdpa_inputs import varlen_lengths
        lens = varlen_lengths(w)
        return (f"{w.name}: packed batch of {len(lens)} sequences ({'+'.join(map(str, lens))} = {w.N} tokens, "
                f"lengths uniform in [{w.len_range[0]}, {w.len_range[1]}]) H={w.H} Hkv={w.Hkv} d={w.d} "
                f"{'causal' if w.causal else 'non-causal'} {'fwd+bwd' if w.with_grad else 'fwd'}")
    if w.kind == "cross":
        what = "fwd+bwd (encoder-decoder cross attention)" if w.with_grad else "fwd (chunked prefill)"
        return (f"{w.name}: B={w.B} H={w.H} Hkv={w.Hkv} Nq={w.n_queries} Nk={w.N} d={w.d} "
                f"{'causal' if w.causal else 'non-causal'} {what}")
    tail = f" (head_dim {w.d_draw} zero-padded)" if w.d_draw else ""
    if w.kind == "fp8":
        tail += " e4m3 inputs (per-tensor scales)"
    return (f"{w.name}: B={w.B} H={w.H} Hkv={w.Hkv} N={w.N} d={w.d}{tail} "
            f"{'causal' if w.causal else 'non-causal'} {'fwd+bwd' if w.with_grad else 'fwd'}")


def step_flops(w):
    from sdpa_inputs import flops_backward, flops_cross, flops_forward
    if w.kind == "masked":
        from sdpa_inputs import flops_masked
        f = flops_masked(w)
        return f, (2.5 * f if w.with_grad else 0.0)
    if w.kind == "varlen":
        from sdpa_inputs import flops_varlen, varlen_lengths
        f = flops_varlen(varlen_lengths(w), w.H, w.d, w.causal)
        return f, (2.5 * f if w.with_grad else 0.0)
    if w.kind == "cross":
        f = flops_cross(w.B, w.H, w.n_queries, w.N, w.d, w.causal)
        return f, (2.5 * f if w.with_grad else 0.0)
    f = flops_forward(w.B, w.H, w.N, w.d, w.causal)
    b = flops_backward(w.B, w.H, w.N, w.d, w.causal) if w.with_grad else 0.0
    return f, b


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def traffic_of(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary profiles/dram_traffic.txt (lines: kernel workload bytes source
    sha1-prefix), or None if absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for ln in lines:
        parts = ln.split()
        if ln.startswith("#") or len(parts) < 5 or parts[0] != kernel or parts[1] != workload:
            continue
        src = os.path.join(ROOT, "scaled_dot_product_08_gb300", "csrc", parts[3])
        try:
            digest = hashlib.sha1(open(src, "rb").read()).hexdigest()[:12]
        except OSError:
            return None
        return float(parts[2]) if parts[4] == digest else None
    return None


class ClockSampler:
    """nvidia-smi samples every 100 ms while running (clocks during the timed region)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float) -> float:
    """Max of a per-rank float over the default process group (identity when
    torch.distributed is not initialised).  NCCL reduces on the GPU, gloo on
    the CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle arm
def _oracle_lengths(w):
    """(query rows, key rows) of the oracle's per-step sample: one head of
    the workload; for a packed batch one head of its first sequence."""
    if w.kind == "varlen":
        from sdpa_inputs import varlen_lengths
        n = varlen_lengths(w)[0]
        return n, n
    return w.n_queries, w.N


def _oracle_head_inputs(w):
    import numpy as np
    from sdpa_inputs import draw
    rng = np.random.default_rng(w.seed)
    dd = w.d_draw or w.d
    nq, nk = _oracle_lengths(w)
    shapes = [(1, 1, nq, dd), (1, 1, nk, dd), (1, 1, nk, dd), (1, 1, nq, dd)]
    return [draw(rng, sh, a) for sh, a in zip(shapes, (w.amp, w.amp, w.amp, 1.0))]


def _oracle_head_seconds(w, x):
    """Wall time of the oracle on one whole head of the workload."""
    import oracle
    q, k, v, do = x
    if w.kind == "masked":
        from sdpa_inputs import prefix_lm_mask, workload_bias
        mask = prefix_lm_mask(w.N, w.prefix) if w.prefix is not None else None
        bias = workload_bias(w)
        t0 = time.perf_counter()
        oracle.attention_masked_forward(q, k, v, w.softmax_scale, w.causal, w.window, None, mask, bias)
        if w.with_grad:
            oracle.attention_masked_backward(q, k, v, do, w.softmax_scale, w.causal, w.window, None, mask, bias)
        return time.perf_counter() - t0
    t0 = time.perf_counter()
    off = (w.N - w.n_queries) if (w.kind == "cross" and w.causal) else 0
    oracle.attention_forward(q, k, v, w.softmax_scale, w.causal, q_offset=off)
    if w.with_grad:
        oracle.attention_backward(q, k, v, do, w.softmax_scale, w.causal, q_offset=off)
    return time.perf_counter() - t0


def _head_flops(w):
    from sdpa_inputs import flops_backward, flops_forward
    if w.kind == "masked":
        from sdpa_inputs import visible_pairs
        return 4.0 * w.d * visible_pairs(w) * (3.5 if w.with_grad else 1.0)
    if w.kind == "varlen":
        n = _oracle_lengths(w)[0]
        return flops_forward(1, 1, n, w.d, w.causal) * (3.5 if w.with_grad else 1.0)
    if w.kind == "cross":
        from sdpa_inputs import flops_cross
        return flops_cross(1, 1, w.n_queries, w.N, w.d, w.causal) * (3.5 if w.with_grad else 1.0)
    return flops_forward(1, 1, w.N, w.d, w.causal) + (flops_backward(1, 1, w.N, w.d, w.causal) if w.with_grad else 0)


def _head_dims(w):
    if w.kind == "varlen":
        return f"N={_oracle_lengths(w)[0]} (its first sequence), d={w.d}"
    n = f"Nq={w.n_queries}, Nk={w.N}" if w.kind == "cross" else f"N={w.N}"
    return f"{n}, d={w.d_draw or w.d}"


def _blas_threads():
    cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        cores = max(i.get("num_threads", 0) for i in threadpool_info()) or cores
    except Exception:
        pass
    return cores


def cpu_baseline(w, budget_s=15.0):
    """fp64 oracle fwd(+bwd) on whole heads of the workload, timed on this
    host's cores (the oracle as it stands), for about `budget_s` seconds."""
    x = _oracle_head_inputs(w)
    done, t_total = 0, 0.0
    while True:
        t_total += _oracle_head_seconds(w, x)
        done += 1
        if t_total >= budget_s or t_total / done * (done + 1) > 2.5 * budget_s:
            break
    return {"value": _head_flops(w) * done / t_total / 1e12, "unit": UNIT, "cores": _blas_threads(),
            "kind": "oracle",
            "sample": f"{done} whole head(s) (B=1, H=1, {_head_dims(w)}) of {w.name}, "
                      f"{'fwd+bwd' if w.with_grad else 'fwd'} in float64 numpy, {t_total:.1f} s"}


def run_reference_decode(args, w):
    """The reference arm for a decode workload: the CPU oracle's decode on
    batch element 0 (all heads, the whole cache) per step, in HBM-equivalent
    bytes per second of the GPU arm's metric."""
    import oracle
    from sdpa_inputs import make_inputs
    x = make_inputs(w)
    q, k, v = x["q"][:1], x["k"][:1], x["v"][:1]
    run = lambda: oracle.attention_decode(q, k, v, w.softmax_scale, w.causal)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    t = time.perf_counter() - t0
    val = decode_bytes(w) / w.B * args.steps / t / 1e9
    sample = f"batch element 0 of {w.name} (all {w.H} heads, Nq={w.n_queries}, Nk={w.N}) per step, float64 numpy"
    line = {"impl": "reference", "metric": "attention decode (KV cache, split over keys) HBM bandwidth",
            "value": val, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded N(0,1) draws rounded to bf16)",
            "config": {"workload": f"{w.name}: B={w.B} H={w.H} Hkv={w.Hkv} Nq={w.n_queries} Nk={w.N} d={w.d} "
                                   f"{'causal' if w.causal else 'non-causal'} decode"},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": _blas_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle, one whole head of the workload per step."""
    if rank != 0:
        return
    if w.kind == "decode":
        run_reference_decode(args, w)
        return
    x = _oracle_head_inputs(w)
    for _ in range(args.warmup):
        _oracle_head_seconds(w, x)
    t = sum(_oracle_head_seconds(w, x) for _ in range(args.steps))
    val = _head_flops(w) * args.steps / t / 1e12
    sample = (f"one whole head (B=1, H=1, {_head_dims(w)}) of {w.name} per step, "
              f"{'fwd+bwd' if w.with_grad else 'fwd'} in float64 numpy")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) draws rounded to bf16)",
            "config": {"workload": workload_desc(w), "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                       "causal": w.causal},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ GPU arm
def run_e2e(torch, sdpa, w, bufs, make_launches, stream, barrier, max_over_ranks, world, flops, Ke):
    """The step end to end from pinned host memory: every step copies its
    inputs host -> device and its outputs (O, lse and, with a backward, dQ,
    dK, dV) device -> host inside the timed region.  The copies are
    pipelined as a data loader would: two slots of device buffers, step i+1's
    inputs going in on one stream and step i-1's outputs coming out on
    another while step i computes on the launching stream."""
    in_keys = ["q", "k", "v"] + (["do"] if w.with_grad else [])
    in_keys += [n for n in ("cu", "mask_t", "bias_t") if bufs[n] is not None]
    out_keys = ["o", "lse"] + (["dq", "dk", "dv"] if w.with_grad else [])
    second = {n: (torch.empty_like(t) if t is not None and n not in ("mask_spec",) else t) for n, t in bufs.items()}
    if bufs["mask_spec"] is not None:
        second["mask_spec"] = sdpa.make_mask(w.window, None, second["mask_t"], w.B, w.H, second["bias_t"])
    slots = [bufs, second]
    launches = [make_launches(b) for b in slots]
    host_in = {n: bufs[n].cpu().pin_memory() for n in in_keys}
    host_out = [{n: torch.empty(b[n].shape, dtype=b[n].dtype).pin_memory() for n in out_keys} for b in slots]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in slots]     # slot's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in slots]   # slot's step has computed
    ev_out = [torch.cuda.Event() for _ in slots]    # slot's outputs are on the host

    def copy_in(i):
        sl = slots[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[i % 2])  # step i - 2 has finished reading the slot
            for n in in_keys:
                sl[n].copy_(host_in[n], non_blocking=True)
            ev_in[i % 2].record(s_in)

    def run(nsteps, start=None, end=None):
        if start is not None:
            start.record(stream)
            s_in.wait_event(start)
        copy_in(0)
        for i in range(nsteps):
            if i + 1 < nsteps:
                copy_in(i + 1)
            stream.wait_event(ev_in[i % 2])
            if i >= 2:
                stream.wait_event(ev_out[i % 2])  # step i - 2's outputs have left the slot
            for launch in launches[i % 2]:
                launch()
            ev_done[i % 2].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i % 2])
                for n in out_keys:
                    host_out[i % 2][n].copy_(slots[i % 2][n], non_blocking=True)
                ev_out[i % 2].record(s_out)
        stream.wait_event(ev_out[(nsteps - 1) % 2])
        stream.wait_event(ev_out[nsteps % 2])
        if end is not None:
            end.record(stream)

    run(2)
    barrier()
    a, bev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(Ke, a, bev)
    barrier()
    ems = max_over_ranks(a.elapsed_time(bev))
    st = sdpa.attn_get_device_status(None)
    if st != 0:
        raise RuntimeError(f"device status after the end-to-end steps: {sdpa.attn_status_string(st)}")
    return {"value": world * flops * Ke / (ems / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ems / Ke, "steps": Ke,
            "note": "inputs in and outputs (O, lse, and dQ, dK, dV with a backward) out every step, pipelined "
                    "with the compute over two buffer slots and two copy streams"}


def run_ours(args, w, rank, world, local_rank):
    import torch
    import scaled_dot_product_08_gb300 as sdpa
    from sdpa_inputs import make_inputs

    sdpa.build()
    sdpa.load()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
    dev = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    B, H, Hkv, N, d = w.B, w.H, w.Hkv, w.N, w.d
    s = w.softmax_scale
    Nq = w.n_queries
    if w.kind == "varlen":
        from sdpa_inputs import make_varlen_inputs
        x = make_varlen_inputs(w)
        cu = torch.from_numpy(x["cu"]).cuda()
        nseq, maxlen = len(x["lengths"]), int(x["lengths"].max())
        lse_shape = (H, N)
    else:
        x = make_inputs(w)
        lse_shape = (B, H, Nq)
    fp8 = None
    if w.kind == "fp8":
        from sdpa_inputs import quantize_e4m3
        fp8 = [quantize_e4m3(x[n]) for n in ("q", "k", "v")]  # (bytes, scale) each
    mask_spec = None
    if w.kind == "masked":
        from sdpa_inputs import prefix_lm_mask, workload_bias
        mask_t = bias_t = None
        if w.prefix is not None:
            mask_t = torch.from_numpy(prefix_lm_mask(N, w.prefix).astype("uint8")).cuda()
        if w.bias_slope is not None:
            bias_t = torch.from_numpy(workload_bias(w)).cuda()
            if w.bias_bf16:
                bias_t = bias_t.to(torch.bfloat16)  # exact: the values are bf16 already
        mask_spec = sdpa.make_mask(w.window, None, mask_t, B, H, bias_t)
        mws_f = sdpa.attn_masked_workspace_size(B, H, Hkv, Nq, N, d, mask_spec, 0)
        mws_b = sdpa.attn_masked_workspace_size(B, H, Hkv, Nq, N, d, mask_spec, 1)
        mws = torch.empty(max(mws_f, mws_b, 16), dtype=torch.uint8, device="cuda")
    if fp8 is not None:
        q, k, v = (torch.from_numpy(b).cuda() for b, _ in fp8)
        o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    else:
        q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
        o = torch.empty_like(q)
    do = dev(x["do"]) if w.with_grad else None
    lse = torch.empty(lse_shape, dtype=torch.float32, device="cuda")
    if w.with_grad:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        if w.kind == "varlen":
            ws_bytes = sdpa.attn_bwd_varlen_workspace_size(nseq, H, Hkv, N, d)
        else:
            ws_bytes = sdpa.attn_bwd_workspace_size(B, H, Hkv, Nq, d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    # The backward: dQ (forming the row vectors D and lse in base 2 on the way),
    # then dK / dV from those vectors.
    names = ["attn_fwd"] + (["attn_bwd_dq", "attn_bwd_grad"] if w.with_grad else [])

    def chk(st, where):
        if st != 0:
            raise RuntimeError(f"{where}: {sdpa.attn_status_string(st)}")

    P = lambda t: t.data_ptr()

    def make_launches(bf):
        """One callable per kernel of the step, in order (names above), on the
        device buffers of `bf` (inputs, outputs, mask)."""
        ptr = lambda n: bf[n].data_ptr() if bf[n] is not None else 0
        pq, pk, pv, po, pl = (ptr(n) for n in ("q", "k", "v", "o", "lse"))
        pdo, pdq, pdk, pdv, pcu = (ptr(n) for n in ("do", "dq", "dk", "dv", "cu"))
        mspec = bf["mask_spec"]
        if w.kind == "varlen":
            def vstage(mask):
                return lambda: chk(sdpa.attn_bwd_varlen_stages(
                    pq, pk, pv, po, pl, pdo, pdq, pdk, pdv, pcu, pcu, P(ws), ws_bytes,
                    nseq, H, Hkv, N, N, maxlen, maxlen, d, s, w.causal, mask, sp), "attn_bwd_varlen_stages")
            launches = [lambda: chk(sdpa.attn_fwd_varlen(pq, pk, pv, po, pl, pcu, pcu, nseq, H, Hkv,
                                                         N, N, maxlen, maxlen, d, s, w.causal, sp), "attn_fwd_varlen")]
            if w.with_grad:
                launches += [vstage(8), vstage(2)]
        elif w.kind == "fp8":
            (_, qsc), (_, ksc), (_, vsc) = fp8
            launches = [lambda: chk(sdpa.attn_fwd_fp8(pq, pk, pv, po, pl, B, H, Hkv, Nq, N, d, s, qsc, ksc,
                                                      vsc, w.causal, sp), "attn_fwd_fp8")]
        elif w.kind == "masked":
            def mstage(mask):
                return lambda: chk(sdpa.attn_bwd_masked_stages(
                    pq, pk, pv, po, pl, pdo, pdq, pdk, pdv, B, H, Hkv, Nq, N, d, s, w.causal,
                    mspec, P(mws), mws.numel(), mask, sp), "attn_bwd_masked_stages")
            launches = [lambda: chk(sdpa.attn_fwd_masked(pq, pk, pv, po, pl, B, H, Hkv, Nq, N, d, s, w.causal,
                                                         mspec, P(mws), mws.numel(), sp), "attn_fwd_masked")]
            if w.with_grad:
                launches += [mstage(8), mstage(2)]
        elif w.kind == "cross":
            launches = [lambda: chk(sdpa.attn_fwd_cross(pq, pk, pv, po, pl, B, H, Hkv, Nq, N, d, s,
                                                        w.causal, sp), "attn_fwd_cross")]
            if w.with_grad:
                launches += [
                    lambda: chk(sdpa.attn_bwd_dq_rows(pq, pk, pv, po, pl, pdo, pdq, P(ws), ws_bytes,
                                                      B, H, Hkv, Nq, N, d, s, w.causal, sp), "attn_bwd_dq_rows"),
                    lambda: chk(sdpa.attn_bwd_grad_cross(pq, pk, pv, pdo, pdk, pdv, P(ws), ws_bytes,
                                                         B, H, Hkv, Nq, N, d, s, w.causal, sp), "attn_bwd_grad_cross")]
        else:
            launches = [lambda: chk(sdpa.attn_fwd(pq, pk, pv, po, pl, B, H, Hkv, N, d, s, w.causal, sp),
                                    "attn_fwd")]
            if w.with_grad:
                launches += [
                    lambda: chk(sdpa.attn_bwd_dq_rows(pq, pk, pv, po, pl, pdo, pdq, P(ws), ws_bytes,
                                                      B, H, Hkv, N, N, d, s, w.causal, sp), "attn_bwd_dq_rows"),
                    lambda: chk(sdpa.attn_bwd_grad(pq, pk, pv, pdo, pdk, pdv, P(ws), ws_bytes,
                                                   B, H, Hkv, N, d, s, w.causal, sp), "attn_bwd_grad")]
        return launches

    bufs = {"q": q, "k": k, "v": v, "o": o, "lse": lse, "do": do, "dq": dq if w.with_grad else None,
            "dk": dk if w.with_grad else None, "dv": dv if w.with_grad else None,
            "cu": cu if w.kind == "varlen" else None, "mask_t": mask_t if w.kind == "masked" else None,
            "bias_t": bias_t if w.kind == "masked" else None, "mask_spec": mask_spec}
    launches = make_launches(bufs)

    # Kernels per step: one per call, plus the mask packing inside the masked
    # forward and first backward calls when there is a boolean mask, and the
    # additive mask's transpose inside the first backward call.
    kernels_per_step = len(launches)
    if w.kind == "masked" and w.prefix is not None:
        kernels_per_step += 2 if w.with_grad else 1
    if w.kind == "masked" and w.bias_slope is not None and w.with_grad:
        kernels_per_step += 1

    def step(evs=None):
        for idx, launch in enumerate(launches):
            if evs is not None:
                evs[idx].record(stream)
            launch()
        if evs is not None:
            evs[len(launches)].record(stream)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # Inputs below twice the L2: evict them before every timed step.
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v) + ((do,) if w.with_grad else ()))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if in_bytes < 2 * L2_BYTES else None

    for _ in range(max(args.warmup, 1)):
        step()
    barrier()
    st = sdpa.attn_get_device_status(None)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {sdpa.attn_status_string(st)}")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        step(evs[i])
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    ms_region = t0.elapsed_time(t1)
    st = sdpa.attn_get_device_status(None)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {sdpa.attn_status_string(st)}")
    per_kernel = {n: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / K for j, n in enumerate(names)}
    # With a flush between steps the step time is the sum of the per-step
    # event spans (first kernel's start to last kernel's end).
    ms = sum(e[0].elapsed_time(e[-1]) for e in evs) if flush is not None else ms_region
    ms = max_over_ranks(ms)
    ms_region = max_over_ranks(ms_region)
    if flush is not None:
        l2_note = (f"flush: a {2 * L2_BYTES / 1e6:.0f} MB buffer is written before each timed step "
                   f"(inputs {in_bytes / 1e6:.0f} MB); step time = sum of per-step event spans")
    else:
        l2_note = f"no flush: inputs ({in_bytes / 1e6:.0f} MB) larger than twice the 129 MB L2"

    f_fwd, f_bwd = step_flops(w)
    flops = f_fwd + f_bwd
    value = world * flops * K / (ms / 1e3) / 1e12

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    dom = max(per_kernel, key=per_kernel.get)
    # Tensor work each kernel executes, in units of one 2*B*H*N^2*d product
    # (halved when causal): the forward runs two (QK^T, PV); the key-tile
    # backward kernel four (S^T, dP^T, dV, dK); the query-tile kernel three
    # (S, dP, dQ).  The step value above keeps the 2.5x-forward convention.
    kflops = {"attn_fwd": f_fwd, "attn_bwd_grad": 2.0 * f_fwd, "attn_bwd_dq": 1.5 * f_fwd}
    achieved = kflops[dom] / (per_kernel[dom] / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    src, nominal = f"{peak_src} bf16 burst (cuBLAS 8192^3)", 2250.0
    if w.kind == "fp8":  # the FP8 peak: the measured bf16 burst times the nominal ratio 4.5 / 2.25
        peak, src, nominal = 2.0 * peak, f"2 x {peak_src} bf16 burst (nominal fp8 / bf16 ratio 4.5 / 2.25)", 4500.0
    roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": src, f"frac_of_nominal_{int(nominal)}": achieved / nominal}
    # Beside the burst peak, the fraction of the measured sustained peak (a
    # seconds-long cuBLAS loop under the power cap), for runs long enough to
    # meet the cap themselves.
    sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    roof["frac_of_sustained"] = achieved / (2.0 * sus if w.kind == "fp8" else sus)
    roof["traffic"] = traffic_of(dom, w.name)
    # The whole step, and the backward, on the method's own FLOPs (forward
    # 4*B*H*N^2*d, halved when causal; backward 2.5 x forward) over the
    # summed kernel times: what the kernels deliver of the work the method
    # needs, whatever they re-execute.
    roof["frac_method_step"] = flops / (sum(per_kernel.values()) / 1e3) / 1e12 / peak
    if w.with_grad:
        roof["frac_method_bwd"] = f_bwd / (sum(per_kernel[n] for n in names[1:]) / 1e3) / 1e12 / peak

    # ---- end to end through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, sdpa, w, bufs, make_launches, stream, barrier, max_over_ranks, world, flops,
                      max(3, min(K, 30)))

    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (fp32 accumulate, bf16 O)" if w.kind == "fp8" else "bf16",
            "data": ("synthetic (seeded N(0,1) draws, quantised per tensor to e4m3)" if w.kind == "fp8"
                     else "synthetic (seeded N(0,1) draws rounded to bf16)"),
            "config": {"workload": workload_desc(w), "B": B, "H": H, "Hkv": Hkv, "N": N, "d": d,
                       "causal": w.causal, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": l2_note},
            "ms_timed_region": ms_region / K,
            "fwd_tflops": f_fwd / (per_kernel["attn_fwd"] / 1e3) / 1e12,
            "kernel_ms": per_kernel,
            "roofline": roof, "cpu_baseline": cb, "e2e": e2e, "clocks": clk,
            "gpu_launches": kernels_per_step * K,
        }
        if w.with_grad:
            line["bwd_tflops"] = f_bwd / (sum(per_kernel[n] for n in names[1:]) / 1e3) / 1e12
        print(json.dumps(line), flush=True)


def decode_bytes(w):
    """Algorithmic HBM bytes of one decode call: read K and V of the cache
    and Q; write O and lse (the chunk partials stay on chip or in L2)."""
    kv = 2 * w.B * w.Hkv * w.N * w.d * 2
    qo = 2 * w.B * w.H * w.n_queries * w.d * 2 + w.B * w.H * w.n_queries * 4
    return kv + qo


def run_decode(args, w, rank, world, local_rank):
    """Decode against a resident KV cache (workloads with Nq set): one step
    is one attn_decode call (chunk pass + merge).  The value is HBM bytes per
    second; e2e copies the step's new queries in and O, lse out (the cache
    stays on the device, as it does across decode steps)."""
    import torch
    import scaled_dot_product_08_gb300 as sdpa
    from sdpa_inputs import make_inputs
    import oracle

    sdpa.build()
    sdpa.load()
    torch.cuda.set_device(local_rank)
    x = make_inputs(w)
    dev = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    B, H, Hkv, Nq, Nk, d = w.B, w.H, w.Hkv, w.n_queries, w.N, w.d
    s = w.softmax_scale
    q = dev(x["q"])
    if w.page_size:
        from sdpa_inputs import paged_layout
        kc, vc, table = paged_layout(w, x["k"], x["v"])
        k, v = dev(kc), dev(vc)
        tbl = torch.from_numpy(table).cuda()
        lens = torch.full((B,), Nk, dtype=torch.int32, device="cuda")
        num_pages, max_pages = kc.shape[0], table.shape[1]
        ws_bytes = sdpa.attn_decode_paged_workspace_size(B, H, Hkv, Nq, w.page_size, max_pages, d)
    else:
        k, v = dev(x["k"]), dev(x["v"])
        ws_bytes = sdpa.attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def step():
        if w.page_size:
            st = sdpa.attn_decode_paged(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        tbl.data_ptr(), lens.data_ptr(), ws.data_ptr(), ws_bytes, B, H, Hkv, Nq,
                                        w.page_size, num_pages, max_pages, d, s, w.causal, sp)
        else:
            st = sdpa.attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  ws.data_ptr(), ws_bytes, B, H, Hkv, Nq, Nk, d, s, w.causal, sp)
        if st != 0:
            raise RuntimeError(f"attn_decode: {sdpa.attn_status_string(st)}")

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(a.elapsed_time(b))
    st = sdpa.attn_get_device_status(None)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {sdpa.attn_status_string(st)}")
    nbytes = decode_bytes(w)
    value = world * nbytes * K / (ms / 1e3) / 1e9
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    per_call = nbytes / (ms / K / 1e3) / 1e9
    roof = {"kernel": ("attn_decode_paged" if w.page_size else "attn_decode") +
                      " (decode_split_kernel + decode_merge_kernel)", "bound": "hbm",
            "achieved": per_call, "peak": peak, "unit": "GB/s", "frac": per_call / peak,
            "peak_source": f"{peak_src} copy bandwidth", "traffic": traffic_of("attn_decode", w.name)}

    e2e = None
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        Ke = max(3, min(K, 50))
        for _ in range(2):
            q.copy_(hq, non_blocking=True); step(); ho.copy_(o, non_blocking=True); hl.copy_(lse, non_blocking=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(Ke):
            q.copy_(hq, non_blocking=True); step(); ho.copy_(o, non_blocking=True); hl.copy_(lse, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(a.elapsed_time(b))
        e2e = {"value": world * nbytes * Ke / (ems / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * 2, "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4,
               "ms_per_step": ems / Ke, "steps": Ke,
               "note": "new queries in, O and lse out; the KV cache stays resident between decode steps"}

    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle as it stands on batch elements, repeated for about 10 s
        done, dt = 0, 0.0
        while dt < 10.0 and done < 200:
            bi = done % B
            t0 = time.perf_counter()
            oracle.attention_decode(x["q"][bi:bi + 1], x["k"][bi:bi + 1], x["v"][bi:bi + 1], s, w.causal)
            dt += time.perf_counter() - t0
            done += 1
        cb = {"value": decode_bytes(w) / B * done / dt / 1e9, "unit": "GB/s", "cores": _blas_threads(), "kind": "oracle",
              "sample": f"{done} batch element(s) of {w.name} (each all {H} heads, Nq={Nq}, Nk={Nk}) in float64 numpy, "
                        f"{dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": "attention decode (KV cache, split over keys) HBM bandwidth", "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) draws rounded to bf16)",
            "config": {"workload": f"{w.name}: B={B} H={H} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} "
                                   f"{'causal' if w.causal else 'non-causal'} decode"
                                   + (f", cache in {w.page_size}-token pages scattered over the pool"
                                      if w.page_size else ""),
                       "B": B, "H": H, "Hkv": Hkv, "Nq": Nq, "Nk": Nk, "d": d, "causal": w.causal,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "no flush: the K/V cache (%.0f MB) is larger than the 129 MB L2" % (2 * B * Hkv * Nk * d * 2 / 1e6)},
            "roofline": roof, "cpu_baseline": cb, "e2e": e2e, "clocks": clk, "gpu_launches": 2 * K,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from sdpa_inputs import workload
    w = workload(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if w.kind == "decode":
            run_decode(args, w, rank, world, local_rank)
        else:
            run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
