#!/usr/bin/env python
"""Throughput of the masked attention backward on GB300.

One step = one attn_bwd call (preprocess, dK/dV, dQ, dSink; plus the mask
tables for block masks) over the workload's full problem, inputs resident in
HBM.  The L2 cache is flushed (a 512 MiB device write) before every timed
step, outside the timed events.  Throughput counts 10*D flops per visible
(b, h, i, j) pair (the five contractions of the backward), so work spent on
masked positions inside partially visible tiles earns nothing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

With N > 1 (launched by torch.distributed.run) every rank runs its own full
copy of the workload (weak scaling: the backward has no exchange step) and the
time is the maximum over ranks.  Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from masked_attention_backward_gb300 import measure  # noqa: E402
from masked_attention_backward_gb300.workloads import BY_NAME, make_inputs  # noqa: E402

METRIC = "attn bwd TFLOP/s over unmasked tiles & ms/call; % of GB300 BF16 tensor peak"
DEFAULT_WORKLOAD = "gqa_sink_causal_s16384"
MASK_NAMES = {0: "none", 1: "causal", 2: "causal+sliding window", 3: "block"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Files whose content decides the dK/dV and dQ kernels' DRAM traffic.
KERNEL_SOURCES = {
    "k_dkdv": ["csrc/attn_kv.cu", "csrc/kv_softmax.cuh", "csrc/tiles.cuh", "csrc/ptx.cuh",
               "csrc/internal.h"],
    "k_dq": ["csrc/attn_dq.cu", "csrc/tiles.cuh", "csrc/ptx.cuh", "csrc/internal.h"],
}


def parse_runs(text: str):
    """--e2e-chunks: "8" (equal runs) or "1,3,3,1" (key/value heads per run)."""
    parts = [int(x) for x in text.split(",")]
    return parts[0] if len(parts) == 1 else parts


def kernel_hash(name: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(name, []):
        with open(os.path.join(ROOT, "masked_attention_backward_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
        except Exception:
            pass
        rows = []
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        if uuid:
            mine = [r for r in rows if uuid.replace("GPU-", "") in r[1]]
            rows = mine or rows
        idx = {r[0] for r in rows}
        if len(idx) > 1:
            rows = [r for r in rows if r[0] == sorted(idx)[0]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        smax = [num(r[3]) for r in rows if num(r[3]) is not None]
        power = [num(r[4]) for r in rows if num(r[4]) is not None]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7),
                              ("sw_thermal_slowdown", 8), ("sw_power_cap", 9)):
                if "Active" in r[col] and "Not" not in r[col]:
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "reasons": sorted(reasons)}


def _pack(x, lens):
    """[B, H, S, D] -> token-major [sum(lens), H, D] (sequence b's first lens[b] rows)"""
    return torch.cat([x[b, :, :L].transpose(0, 1) for b, L in enumerate(lens)], dim=0).contiguous()


def gpu_inputs(wl, device, packed=False):
    """Device inputs of a workload; O and LSE from the CUDA forward.  packed:
    a variable-length workload in the packed layout (token-major tensors and
    cumulative sequence offsets) instead of the padded BHSD one."""
    from masked_attention_backward_gb300 import binding as mab
    inp = make_inputs(wl)
    sink = inp.sink.to(device) if inp.sink is not None else None
    bm = inp.block_mask.to(device) if inp.block_mask is not None else None
    if packed:
        lq = [int(x) for x in inp.seqlen_q]
        lk = [int(x) for x in inp.seqlen_k]
        q, dO = (_pack(t, lq).to(device) for t in (inp.q, inp.dO))
        k, v = (_pack(t, lk).to(device) for t in (inp.k, inp.v))
        mask = mab.packed_mask(wl.mask_kind, lq, lk, device, window=wl.window, bx=wl.bx,
                               by=wl.by, block_mask=bm)
        o, lse = mab.fwd(q, k, v, sink, mask, wl.scale)
        torch.cuda.synchronize()
        return inp, dict(q=q, k=k, v=v, o=o, dO=dO, lse=lse, sink=sink, mask=mask)
    q, k, v, dO = (t.to(device) for t in (inp.q, inp.k, inp.v, inp.dO))
    lq = inp.seqlen_q.to(device) if inp.seqlen_q is not None else None
    lk = inp.seqlen_k.to(device) if inp.seqlen_k is not None else None
    mask = mab.Mask(kind=wl.mask_kind, window=wl.window, bx=wl.bx, by=wl.by, block_mask=bm,
                    seqlen_q=lq, seqlen_k=lk)
    o, lse = mab.fwd(q, k, v, sink, mask, wl.scale)   # O and LSE from the CUDA forward
    torch.cuda.synchronize()
    return inp, dict(q=q, k=k, v=v, o=o, dO=dO, lse=lse, sink=sink, mask=mask)


def run_ours(args, rank, world, local):
    from masked_attention_backward_gb300 import binding as mab
    mab.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = BY_NAME[args.workload]
    inp, t = gpu_inputs(wl, device)
    pairs = measure.visible_pairs(wl, inp.block_mask, inp.seqlen_q, inp.seqlen_k)
    fl = measure.flops(wl, pairs)
    ws = mab.workspace(mab.shape_of(t["q"], t["k"]), t["mask"], device)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    dsink = torch.empty_like(t["sink"]) if t["sink"] is not None else None
    out = (dq, dk, dv, dsink)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)

    def step():
        mab.bwd(t["q"], t["k"], t["v"], t["o"], t["dO"], t["lse"], t["sink"], t["mask"],
                wl.scale, ws=ws, out=out, compensated=args.compensated)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    status = mab.device_status(ws)
    if status != mab.ATTN_OK:
        raise RuntimeError("device status after warm-up: " + mab.attn_status_string(status))

    # ---- device-timed steps (the library's per-kernel events stay off here:
    # they would sit between the kernels and keep dQ from starting on the SMs
    # that the dK/dV grid's last CTAs leave idle)
    clocks = ClockSampler(local).start()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()

    # ---- per-kernel breakdown: a separate pass with the library's events on
    mab.attn_profile_enable(True)
    kern = {}
    per_step_launches = 0
    for _ in range(min(args.steps, 20)):
        flush.zero_()
        step()
        torch.cuda.synchronize()
        prof = mab.attn_profile_read()
        per_step_launches = len(prof)
        for name, ms in prof:
            kern.setdefault(name, []).append(ms)
    mab.attn_profile_enable(False)
    launches = per_step_launches * args.steps  # our kernels in the timed region
    status = mab.device_status(ws)
    if status != mab.ATTN_OK:
        raise RuntimeError("device status after timing: " + mab.attn_status_string(status))
    t_rank = float(sum(step_ms))
    t_max = max_over_ranks(t_rank, world, device)
    ms_per_step = t_max / args.steps
    value = world * fl["total"] * args.steps / (t_max * 1e-3) / 1e12

    # ---- end to end from pinned host buffers: every step copies its inputs in
    # and its gradients out; the binding overlaps the copies of one run of GQA
    # groups with the kernels of the previous one (each run is one attn_bwd call)
    e2e = None
    if not args.no_e2e:
        host_in = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "o", "dO", "lse")}
        host_in["sink"] = t["sink"].cpu().pin_memory() if t["sink"] is not None else None
        host_out = [x.cpu().pin_memory() if x is not None else None for x in out]
        hb = mab.HostBackward(wl.B, wl.Hq, wl.Hkv, wl.Sq, wl.Skv, t["q"].dtype, t["mask"],
                              wl.scale, t["sink"] is not None, device, chunks=args.e2e_chunks,
                              compensated=args.compensated)
        h2d, d2h = hb.bytes_per_call(host_in, host_out)
        e2e_ms = []
        for it in range(args.warmup + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            hb(host_in, host_out)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
        te = max_over_ranks(float(sum(e2e_ms)), world, device)
        e2e = {"value": round(world * fl["total"] * args.steps / (te * 1e-3) / 1e12, 2),
               "unit": "TFLOP/s", "ms_per_step": round(te / args.steps, 3),
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipeline_chunks": hb.chunks, "pipeline_runs": hb.sizes}
        # the same gradients as the device-resident calls timed above
        for a, b_ in zip(host_out, out):
            if a is not None and not torch.equal(a, b_.cpu()):
                raise RuntimeError("pipelined host-buffer backward differs from attn_bwd")

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    avg = {n: float(np.mean(v)) for n, v in kern.items()}
    dom = max(("k_dkdv", "k_dq"), key=lambda n: avg.get(n, 0.0))
    dom_flops = fl["dkdv"] if dom == "k_dkdv" else fl["dq"]
    achieved = dom_flops / (avg[dom] * 1e-3) / 1e12
    # the kernels run inside steps of about 10 ms (the timed region lasts about
    # a second), where the SM clock stays near its maximum: the burst cuBLAS
    # rate is the comparable peak; fp16 and bf16 share the dense tensor rate
    peak = peaks.get("bf16_tflops") or peaks.get("bf16_tflops_sustained")
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tr = json.load(f)
        ent = tr.get(args.workload, {}).get(dom)
        if ent and ent.get("source_hash") == kernel_hash(dom):
            traffic = ent.get("bytes_per_launch")
    kernels = {}
    for n, a in avg.items():
        d = {"ms": round(a, 4), "share": round(sum(kern[n]) / sum(sum(v) for v in kern.values()), 4)}
        if n == "k_dkdv":
            d["tflops"] = round(fl["dkdv"] / (a * 1e-3) / 1e12, 1)
        elif n == "k_dq":
            d["tflops"] = round(fl["dq"] / (a * 1e-3) / 1e12, 1)
        elif n == "k_preprocess":
            d["gbps"] = round(measure.algorithmic_bytes(wl, 0, inp.seqlen_q, inp.seqlen_k)
                              ["preprocess"] / (a * 1e-3) / 1e9, 1)
        kernels[n] = d

    # ---- the forward that produced O and LSE, timed on its own (not part of
    # the step): same inputs, L2 flushed before every call
    fwd_ms = []
    for it in range(3 + min(args.steps, 20)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mab.fwd(t["q"], t["k"], t["v"], t["sink"], t["mask"], wl.scale, ws=ws)
        e1.record(stream)
        e1.synchronize()
        if it >= 3:
            fwd_ms.append(e0.elapsed_time(e1))
    f_ms = float(np.median(fwd_ms))
    forward = {"ms": round(f_ms, 4), "tflops": round(fl["fwd"] / (f_ms * 1e-3) / 1e12, 1),
               "calls": len(fwd_ms), "flops_per_call": fl["fwd"],
               "note": "attn_fwd (O, LSE) on the step's inputs; median of the calls, "
                       "outside the timed step"}

    table = None
    if not args.no_workloads:
        table = {}
        for name, bound in TABLE_WORKLOADS:
            if name != args.workload:
                table[name] = time_workload(name, bound, device, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, inp, fl, budget_s=args.cpu_seconds)
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": dict(workload_config(wl, pairs, fl, inp),
                       **({"compensated": True} if args.compensated else {})),
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst cuBLAS bf16 GEMM; the "
                                    f"kernel is timed inside steps of ~10 ms at the clocks "
                                    f"reported in 'clocks')",
                     "flops_per_launch": dom_flops},
        "kernels": kernels,
        "forward": forward,
        "pct_of_peak_end_to_end": round(value / world / peak, 4),
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if table is not None:
        line["workloads"] = table
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


# The other named workloads, timed after the headline one and reported beside it
# (one row each): the tiny sliding-window case (launch-latency bound: reported
# in microseconds), the 4096-token sliding window and the bigbird block mask
# (both bound by HBM traffic: achieved GB/s of algorithmic bytes against the
# measured copy bandwidth), the random 30 % block mask (tensor-bound), and the
# variable-length batch.
TABLE_WORKLOADS = [
    ("gqa_sink_swa64_tiny", "latency"),
    ("gqa_sink_swa128_s4096", "hbm"),
    ("blocksparse_random30_s8192", "tensor"),
    ("blocksparse_bigbird_5000x7000", "hbm"),
    ("gqa_sink_varlen_causal_b8_s2048", "tensor"),
    ("gqa_sink_varlen_causal_b8_s2048_packed", "tensor"),
    # the single-pass design (dq partials + fixed-order reduction) beside the
    # split one, on the workloads whose walks are short
    ("gqa_sink_swa128_s4096_single_pass", "hbm"),
    ("blocksparse_random30_s8192_single_pass", "tensor"),
    ("blocksparse_bigbird_5000x7000_single_pass", "hbm"),
    ("gqa_sink_varlen_causal_b8_s2048_single_pass", "tensor"),
]
PACKED_SUFFIX = "_packed"
SINGLE_PASS_SUFFIX = "_single_pass"


def time_workload(name, bound, device, peaks, min_steps=20, min_seconds=0.6, max_steps=2000):
    """One row of the per-workload table: warm-up, then steps (L2 flushed before
    each, outside the events) until at least min_seconds of wall time have
    passed, with nvidia-smi sampling the clocks; then up to 20 steps with the
    library's per-kernel events on."""
    from masked_attention_backward_gb300 import binding as mab
    packed = name.endswith(PACKED_SUFFIX)
    single = name.endswith(SINGLE_PASS_SUFFIX)
    base = name[:-len(PACKED_SUFFIX)] if packed else name
    base = base[:-len(SINGLE_PASS_SUFFIX)] if single else base
    wl = BY_NAME[base]
    inp, t = gpu_inputs(wl, device, packed=packed)
    pairs = measure.visible_pairs(wl, inp.block_mask, inp.seqlen_q, inp.seqlen_k)
    fl = measure.flops(wl, pairs)
    ab = measure.algorithmic_bytes(
        wl, 0 if inp.block_mask is None else int(inp.block_mask.numel()), inp.seqlen_q,
        inp.seqlen_k)
    flags = mab.ATTN_FLAG_SINGLE_PASS if single else 0
    ws = mab.workspace(mab.shape_of(t["q"], t["k"], flags, mask=t["mask"]), t["mask"], device)
    out = (torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"]),
           torch.empty_like(t["sink"]) if t["sink"] is not None else None)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)

    def step():
        mab.bwd(t["q"], t["k"], t["v"], t["o"], t["dO"], t["lse"], t["sink"], t["mask"],
                wl.scale, ws=ws, out=out, single_pass=single)

    for _ in range(5):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index or 0).start()
    ms = []
    w0 = time.perf_counter()
    while len(ms) < max_steps and (len(ms) < min_steps or time.perf_counter() - w0 < min_seconds):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    clk = clocks.stop()
    mab.attn_profile_enable(True)
    kern = {}
    for _ in range(20):
        flush.zero_()
        step()
        torch.cuda.synchronize()
        for kname, kms in mab.attn_profile_read():
            kern.setdefault(kname, []).append(kms)
    mab.attn_profile_enable(False)
    status = mab.device_status(ws)
    if status != mab.ATTN_OK:
        raise RuntimeError(f"{name}: device status " + mab.attn_status_string(status))
    med = float(np.median(ms))
    tflops = fl["total"] / (med * 1e-3) / 1e12
    gbps = ab["total"] / (med * 1e-3) / 1e9
    tpk = peaks.get("bf16_tflops") or peaks.get("bf16_tflops_sustained")
    row = {"ms": round(med, 4), "us": round(med * 1e3, 1),
           "ms_p10": round(float(np.percentile(ms, 10)), 4),
           "ms_p90": round(float(np.percentile(ms, 90)), 4), "steps": len(ms),
           "tflops": round(tflops, 1), "frac_tensor_end_to_end": round(tflops / tpk, 4),
           "alg_bytes": int(ab["total"]), "gbps_alg": round(gbps, 1),
           "frac_hbm": round(gbps / peaks["hbm_gbs"], 4), "bound": bound,
           "dtype": wl.dtype, "config": dict(workload_config(wl, pairs, fl, inp),
                                             **({"layout": "packed (token-major tensors, "
                                                           "cumulative sequence offsets)"}
                                                if packed else {}),
                                             **({"design": "single pass (dq partials in the "
                                                           "workspace, fixed-order reduction)",
                                                 "workspace_gb": round(ws.numel() / 1e9, 3)}
                                                if single else {})),
           "clocks": clk}
    kd = {}
    for kname, v in kern.items():
        a = float(np.mean(v))
        d = {"ms": round(a, 4)}
        if kname == "k_dkdv":
            d["tflops"] = round(fl["dkdv"] / (a * 1e-3) / 1e12, 1)
            d["frac"] = round(d["tflops"] / tpk, 4)
        elif kname == "k_dq":
            d["tflops"] = round(fl["dq"] / (a * 1e-3) / 1e12, 1)
            d["frac"] = round(d["tflops"] / tpk, 4)
        elif kname == "k_dkdvq":
            # all five contractions of the visible pairs
            d["tflops"] = round(fl["total"] / (a * 1e-3) / 1e12, 1)
            d["frac"] = round(d["tflops"] / tpk, 4)
        elif kname == "k_preprocess":
            d["gbps"] = round(ab["preprocess"] / (a * 1e-3) / 1e9, 1)
        kd[kname] = d
    row["kernels"] = kd
    row["kernels_note"] = ("per-kernel events serialise the kernels (the dQ grid then cannot "
                           "start on SMs the dK/dV grid's tail leaves idle), so their sum "
                           "exceeds ms")
    return row


def workload_config(wl, pairs, fl, inp=None):
    cfg = _workload_config(wl, pairs, fl)
    if inp is not None and inp.seqlen_q is not None:
        cfg["seqlen_q"] = [int(x) for x in inp.seqlen_q]
        cfg["seqlen_k"] = [int(x) for x in inp.seqlen_k]
        cfg["varlen"] = (f"per-batch valid lengths, uniform in [{math.ceil(wl.varlen_min * wl.Sq)},"
                         f" {wl.Sq}], on the padded BHSD layout")
    return cfg


def _workload_config(wl, pairs, fl):
    return {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "Sq": wl.Sq,
            "Skv": wl.Skv, "D": wl.D, "mask": MASK_NAMES[wl.mask_kind],
            "window": wl.window or None, "bx": wl.bx if wl.mask_kind == 3 else None,
            "by": wl.by if wl.mask_kind == 3 else None, "sink": wl.sink,
            "visible_pairs": int(pairs), "flops_per_step": int(fl["total"]),
            "l2": "flushed before every step (512 MiB device write, outside the timed events)",
            "o_lse_source": "CUDA forward (attn_fwd) on the same inputs"}


def cpu_baseline(wl, inp, fl, budget_s: float = 15.0, seed: int = 0):
    """Time the fp64 oracle on a bounded random sample of query rows (dQ) and
    key rows (dK, dV) of the workload and extrapolate to one full call.

    The oracle's cost per row does not depend on the values of O and LSE, so
    the sample runs with placeholder statistics (LSE = 0, Delta = 0)."""
    import oracle
    rng = np.random.default_rng(seed)
    pb = oracle.Problem(B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, Sq=wl.Sq, Skv=wl.Skv, D=wl.D,
                        scale=wl.scale, mask_kind=wl.mask_kind, window=wl.window, bx=wl.bx,
                        by=wl.by,
                        block_mask=None if inp.block_mask is None else inp.block_mask.numpy(),
                        sink=None if inp.sink is None else inp.sink.double().numpy(),
                        seqlen_q=None if inp.seqlen_q is None else inp.seqlen_q.numpy(),
                        seqlen_k=None if inp.seqlen_k is None else inp.seqlen_k.numpy())
    q = inp.q.double().numpy()
    k = inp.k.double().numpy()
    v = inp.v.double().numpy()
    dO = inp.dO.double().numpy()
    lse = np.zeros((wl.B, wl.Hq, wl.Sq))
    dl = np.zeros((wl.B, wl.Hq, wl.Sq))
    nrows, ncols = wl.B * wl.Hq * wl.Sq, wl.B * wl.Hkv * wl.Skv
    per = {"rows": 0.0, "cols": 0.0}
    counts = {"rows": 0, "cols": 0}
    n = 4
    t_start = time.perf_counter()
    while True:
        rows = rng.integers(0, nrows, size=n)
        cols = rng.integers(0, ncols, size=max(1, n // 8))
        t0 = time.perf_counter()
        oracle.dq_rows(pb, q, k, v, dO, lse, dl, rows)
        t1 = time.perf_counter()
        oracle.dkdv_cols(pb, q, k, v, dO, lse, dl, cols)
        t2 = time.perf_counter()
        per["rows"] += t1 - t0
        per["cols"] += t2 - t1
        counts["rows"] += rows.size
        counts["cols"] += cols.size
        spent = time.perf_counter() - t_start
        if spent >= budget_s:
            break
        n = int(min(n * 2, max(4, n * (budget_s - spent) / max(t2 - t0, 1e-3))))
    est = per["rows"] / counts["rows"] * nrows + per["cols"] / counts["cols"] * ncols
    return {"value": round(fl["total"] / est / 1e12, 6), "unit": "TFLOP/s",
            "ms_per_call": round(est * 1e3, 1), "extrapolated": True,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{counts['rows']} random query rows (dQ) and {counts['cols']} random key "
                      f"rows (dK, dV) of {wl.name}, fp64, {round(time.perf_counter() - t_start, 1)}"
                      f" s of CPU time, extrapolated to the full call by row counts"}


def run_reference(args, rank, world):
    """The fp64 oracle as the reference arm: rank 0 only, host cores."""
    if rank != 0:
        return None
    wl = BY_NAME[args.workload]
    inp = make_inputs(wl)
    pairs = measure.visible_pairs(wl, inp.block_mask, inp.seqlen_q, inp.seqlen_k)
    fl = measure.flops(wl, pairs)
    per_step = max(2.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    per_step = min(per_step, args.cpu_seconds)   # --cpu-seconds bounds each sample
    for i in range(args.warmup):
        cpu_baseline(wl, inp, fl, budget_s=per_step / 4, seed=100 + i)
    ests = [cpu_baseline(wl, inp, fl, budget_s=per_step, seed=i) for i in range(args.steps)]
    ms = float(np.mean([e["ms_per_call"] for e in ests]))
    value = fl["total"] / (ms * 1e-3) / 1e12
    cpu = dict(ests[-1])
    cpu["value"] = round(value, 6)
    cpu["sample"] = f"{args.steps} timed samples; last: " + cpu["sample"]
    cpu["extrapolated"] = True
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 1), "extrapolated": True,
            "extrapolation": "each step times the oracle on a bounded random sample of rows "
                             "and scales to one full call by row counts; ms_per_step is that "
                             "estimate, not a measured wall time",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, pairs, fl, inp), "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(BY_NAME))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload table timed after the headline workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--compensated", action="store_true",
                    help="time the compensated backward (P and dS as high part + remainder)")
    ap.add_argument("--e2e-chunks", type=parse_runs, default=8,
                    help="runs of GQA groups the host-buffer pipeline overlaps: a count of "
                         "equal runs, or the key/value heads of each run (e.g. 1,3,3,1)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
