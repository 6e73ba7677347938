#!/usr/bin/env python
"""Benchmark of exact response-replay attention (one GRPO group replay over a
captured, paged long prompt) on GB300.

One step = capture-side page write of the whole prompt (A1) + serial replay of
the G group members (A2-A8: forward, preprocess, backward of each member into
one reused workspace).  Metric: algorithmic replay flops per second
(forward 4 + backward 6 times R*P*d*Hq for the prompt part, 4 + 10 times
d*Hq*R(R+1)/2 for the causal response part), with prompt-KV GB/s and replays/s
alongside.  Default workload: 2,097,152-position prompt in 8192 pages of 256,
24/4 heads, d=256, G=8 members of 4096 tokens, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the float64 CPU oracle arm
    python bench.py --workload prefill_bf16_p256k   # the capture step, ls_prompt_prefill

Under torchrun each rank runs its own replica of the workload (members are
independent; no data-path collective), the timing is the max over ranks and
value is the whole-job aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "replay attn fwd+bwd TFLOP/s and prompt-KV GB/s at 2M-token prefix; replays/s"
DEFAULT_WORKLOAD = "bf16_p2m_r4096_g8"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def replay_flops(P, R, hq, d):
    return 10.0 * R * P * d * hq + 14.0 * d * hq * R * (R + 1) / 2.0


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.f.flush()
        rows = []
        try:
            for line in open(self.f.name):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        finally:
            os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


def recorded_traffic(kernel: str, workload: str, source_file: Path):
    """Per-launch DRAM bytes recorded by an ncu capture in profiles/ for this
    kernel and workload, or None when absent or taken on another source."""
    p = ROOT / "profiles" / f"{kernel}_{workload}.md"
    if not p.exists():
        return None
    sha = hashlib.sha256(source_file.read_bytes()).hexdigest()[:16]
    vals = {}
    for line in p.read_text().splitlines():
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_sha")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != sha or "traffic_bytes_per_launch" not in vals:
        return None
    return float(vals["traffic_bytes_per_launch"])


def max_over_ranks(ms: float, device) -> float:
    """Slowest rank's time: the whole job is done when every replica is."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replay_config(workload: str, w, world: int, host_pages: int = 0, member_major: bool = False) -> dict:
    """The config object of a replay line; both arms print the same one."""
    kv_bytes_pass = w.prompt_len * w.hkv * w.head_dim * 2 * (2 if w.dtype == "bf16" else 4)
    order = ("one member at a time" if member_major else
             "chunk-major: each pass streams the prompt once for the group")
    return {"workload": workload, "prompt_len": w.prompt_len, "resp_lens": list(w.resp_lens),
            "group": w.group, "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim,
            "page_size": w.page_size, "parallelism": f"replicas x{world}",
            "pages": ("HBM" if host_pages <= 0 else
                      f"pinned host memory, streamed in chunks of {host_pages} pages, {order} "
                      "(capture outside the timed steps)"),
            "l2": "inputs larger than L2 (prompt K/V %.1f GiB per pass)" % (kv_bytes_pass / 2**30)}


def clock_matched(roof: dict, pk: dict, clocks: dict) -> None:
    """Adds to a tensor-bound roofline the peak rescaled from the clock the
    peak was measured at to the median SM clock of this run (the tensor pipe
    does a fixed amount of work per clock), and the launch time in clocks."""
    ref_mhz = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    mhz = clocks.get("sm_mhz")
    if mhz:
        roof["launch_kcycles"] = round(roof["launch_ms"] * mhz, 1)
    if roof.get("bound") != "tensor" or not ref_mhz or not mhz:
        return
    peak = roof["peak"] * mhz / ref_mhz
    roof["clock_matched"] = {"peak": round(peak, 1), "frac": roof["achieved"] / peak,
                             "sm_mhz": mhz, "peak_sm_mhz": ref_mhz}


def job_throughput(flops_per_rank_step: float, world: int, ms_step: float) -> float:
    """Whole-job TFLOP/s: every rank processes its own replica (weak scaling)."""
    return flops_per_rank_step * world / (ms_step * 1e-3) / 1e12


# --------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    import long_context_grpo_replay_gb300.binding as ls
    from long_context_grpo_replay_gb300 import build, inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    ls.lib()
    w = inputs.WORKLOADS[args.workload]
    G, P, d, hq, hkv = w.group, w.prompt_len, w.head_dim, w.hq, w.hkv
    tdt = inputs.torch_dtype(w)
    desc = ls.desc_for(hq, hkv, d, w.page_size, tdt, w.scale)

    # ---- device-resident inputs (seeded synthetic, generated on the device)
    src = inputs.make_prompt_source(w.with_(seed=w.seed + 1000 * rank), dev)
    pool_shape = (w.pool_pages, hkv, w.page_size, d)
    k_pool = torch.empty(pool_shape, dtype=tdt, device=dev)
    v_pool = torch.empty(pool_shape, dtype=tdt, device=dev)
    pt = src["page_table"]
    prompt = ls.prompt_from(k_pool, v_pool, pt, P)
    members = []
    for g in range(G):
        m = inputs.make_member(w.with_(seed=w.seed + 1000 * rank), g, dev)
        R = m["q"].shape[0]
        m.update(o=torch.empty_like(m["q"]), lse=torch.empty(R, hq, device=dev, dtype=torch.float32),
                 delta=torch.empty(R, hq, device=dev, dtype=torch.float32),
                 dq=torch.empty_like(m["q"]),
                 dk=torch.empty_like(m["k"]), dv=torch.empty_like(m["v"]))
        members.append(m)
    ws = torch.empty(ls.ls_replay_workspace_size(desc, prompt, max(w.resp_lens)),
                     dtype=torch.uint8, device=dev)
    ls.ls_clear_device_status(ws)
    stream = torch.cuda.current_stream(dev)

    def step():
        ls.ls_kv_page_write(desc, k_pool, v_pool, pt, 0, src["k"], src["v"], ws, stream)
        ls.ls_replay_group(desc, prompt, members, ws, stream)

    host = None
    if args.host_pages > 0:
        # pages resident in pinned host memory, streamed in chunks each pass;
        # written once into the host pool (capture, outside the timed steps)
        from long_context_grpo_replay_gb300.host_pages import HostPagedReplay

        ls.ls_kv_page_write(desc, k_pool, v_pool, pt, 0, src["k"], src["v"], ws, stream)
        torch.cuda.synchronize()
        kh = k_pool.cpu().pin_memory()
        vh = v_pool.cpu().pin_memory()
        host = HostPagedReplay(desc, kh, vh, pt.cpu(), P, args.host_pages, dev)
        ws = torch.empty(host.workspace_bytes(max(w.resp_lens)), dtype=torch.uint8, device=dev)
        ls.ls_clear_device_status(ws)

        if args.host_pages_member_major:
            def step():
                for m in members:
                    host.forward(m["q"], m["k"], m["v"], m["o"], m["lse"], ws)
                    host.backward(m["q"], m["k"], m["v"], m["d_o"], m["o"], m["lse"], m["dq"],
                                  m["dk"], m["dv"], ws)
        else:
            def step():  # chunk-major: each pass streams the prompt once for the group
                host.forward_group(members, ws)
                host.backward_group(members, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)

    # ---- timed region: K steps, events on the launching stream
    ls.ls_trace_enable(True)
    ls.ls_trace_reset()
    launches0 = ls.ls_launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # one event between consecutive steps as well, for the per-step median
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for i in range(args.steps):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = ls.ls_launch_count() - launches0
    ms_total = ev[0].elapsed_time(ev[-1])
    ms_median = statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps))
    trace = ls.kernel_trace()
    ls.ls_trace_enable(False)
    ls.ls_read_device_status(ws)
    clocks = clk.summary()
    memory = {  # the workspace is sized for the longest member, not for G
        "peak_allocated_gib": round(torch.cuda.max_memory_allocated(dev) / 2**30, 2),
        "workspace_gib": round(ws.numel() / 2**30, 3),
        "member_io_gib": round(sum(t.numel() * t.element_size() for m in members for t in m.values())
                               / G / 2**30, 3),
    }
    ms_total = max_over_ranks(ms_total, dev)
    ms_median = max_over_ranks(ms_median, dev)
    ms_step = ms_total / args.steps
    flops_step = sum(replay_flops(P, R, hq, d) for R in w.resp_lens)
    value = job_throughput(flops_step, world, ms_step)
    kv_bytes_pass = P * hkv * d * 2 * (2 if tdt == torch.bfloat16 else 4)
    kv_gbs = 2 * G * kv_bytes_pass * world / (ms_step * 1e-3) / 1e9
    # the same with each member's own tensors counted once per pass that
    # touches them: forward Q, K_r, V_r in, O and LSE out; preprocess O, dO in,
    # D out; backward Q, K_r, V_r, dO, LSE, D in, dQ, dK, dV out
    esz = 2 if tdt == torch.bfloat16 else 4
    io_member = sum((7 * R * hq * d + 6 * R * hkv * d) * esz + 4 * R * hq * 4 for R in w.resp_lens)
    kv_io_gbs = (2 * G * kv_bytes_pass + io_member) * world / (ms_step * 1e-3) / 1e9

    # ---- roofline of the dominant kernel (time from the traced events)
    pk, pk_src = peaks()
    dom = max(("tc_fwd", "tc_bwd_dq", "simt_fwd", "simt_bwd_dq"),
              key=lambda k: trace.get(k, (0, 0.0))[1])
    n_l, t_l = trace.get(dom, (0, 0.0))
    # one launch per member, or one per staged chunk with host pages: the
    # roofline is taken per member either way
    per_launch_ms = t_l / max(1, n_l) if host is None else t_l / (G * args.steps)
    coef = 4.0 if dom.endswith("fwd") else 6.0
    flops_launch = sum(coef * R * P * d * hq for R in w.resp_lens) / G
    bytes_launch = kv_bytes_pass
    # the bound is the one the kernel's arithmetic intensity (flop per
    # prompt-K/V byte) puts it under: tensor above the ridge of the measured
    # peaks, HBM below it
    peak_t = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_m = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ridge = peak_t * 1e12 / (peak_m * 1e9)
    if flops_launch / bytes_launch >= ridge:
        achieved = flops_launch / (per_launch_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                "frac": achieved / peak_t}
    else:
        achieved = bytes_launch / (per_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak_m, "unit": "GB/s",
                "frac": achieved / peak_m}
    src_file = ROOT / "long_context_grpo_replay_gb300" / "csrc" / (
        "ls_tc_fwd.cu" if dom == "tc_fwd" else "ls_tc_bwd.cu" if dom == "tc_bwd_dq" else "ls_simt.cu")
    roof["traffic"] = recorded_traffic(dom, args.workload, src_file)
    roof["kernel"] = dom
    roof["peak_source"] = f"{pk_src} ({'bf16_tflops_sustained' if roof['bound'] == 'tensor' else 'hbm_gbs'})"
    roof["algorithmic_per_launch"] = flops_launch if roof["bound"] == "tensor" else bytes_launch
    roof["launch_ms"] = per_launch_ms
    clock_matched(roof, pk, clocks)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and host is None:
        e2e = run_e2e(args, w, desc, src, members, k_pool, v_pool, pt, prompt, ws, stream, dev,
                      flops_step, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, k_pool, v_pool, pt, members, budget_s=args.cpu_budget)

    # the pages' second regime (short responses over the same 2M prefix) and
    # their memory property (peak memory nearly flat in G), in this process
    short = mem_g = None
    if args.workload == DEFAULT_WORKLOAD and host is None and not args.no_extras:
        short = short_response_leg(args, desc, prompt, ws, stream, dev, pk, clocks)
        del src, members
        mem_g = memory_vs_group(w, desc, prompt, ws, stream, dev)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1)/sqrt(d) Q/K/V, N(0,1) dO, random page table)",
            "config": replay_config(args.workload, w, world,
                                    args.host_pages if host is not None else 0,
                                    args.host_pages_member_major),
            "prompt_kv_gbs": round(kv_gbs, 1),
            "prompt_kv_and_member_io_gbs": round(kv_io_gbs, 1),
            "replays_per_s": round(G * world / (ms_step * 1e-3), 4),
            "replays_per_s_median_step": round(G * world / (ms_median * 1e-3), 4),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "memory": memory,
            "kernels_ms_per_step": {k: round(v[1] / args.steps, 3) for k, v in trace.items()},
        }
        if short is not None:
            line["short_response"] = short
        if mem_g is not None:
            line["memory_vs_group"] = mem_g
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


SHORT_WORKLOAD = "bf16_p2m_r64_g8"


def short_response_leg(args, desc, prompt, ws, stream, dev, pk, clocks):
    """The KV-streaming regime: G=8 members of 64 tokens over the 2M-position
    prompt pages already written, timed (steps x group replay, after the
    warm-up) with CUDA events on the stream.  Reports the forward's and the
    backward's prompt-K/V GB/s and their fractions of the HBM and tensor
    peaks (with each kernel's DRAM bytes per launch when an ncu capture of
    the current source is recorded), next to the ceiling the arithmetic
    intensity allows: at R = 64 a
    prompt-K/V byte carries 384 flop in the forward and 576 in the backward,
    above the ridge of the measured peaks, so the tensor pipe, not HBM, is the
    first limit."""
    import torch

    import long_context_grpo_replay_gb300.binding as ls
    from long_context_grpo_replay_gb300 import inputs

    w = inputs.WORKLOADS[SHORT_WORKLOAD]
    G, P, d, hq, hkv = w.group, w.prompt_len, w.head_dim, w.hq, w.hkv
    members = []
    for g in range(G):
        m = inputs.make_member(w, g, dev)
        R = m["q"].shape[0]
        m.update(o=torch.empty_like(m["q"]), lse=torch.empty(R, hq, device=dev, dtype=torch.float32),
                 delta=torch.empty(R, hq, device=dev, dtype=torch.float32),
                 dq=torch.empty_like(m["q"]), dk=torch.empty_like(m["k"]), dv=torch.empty_like(m["v"]))
        members.append(m)
    for _ in range(args.warmup):
        ls.ls_replay_group(desc, prompt, members, ws, stream)
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)
    ls.ls_trace_enable(True)
    ls.ls_trace_reset()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n = max(3, args.steps)
    e0.record(stream)
    for _ in range(n):
        ls.ls_replay_group(desc, prompt, members, ws, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    trace = ls.kernel_trace()
    ls.ls_trace_enable(False)
    ls.ls_read_device_status(ws)
    ms = e0.elapsed_time(e1) / n
    peak_t = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_m = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kv = P * hkv * d * 2 * 2
    ridge = peak_t * 1e12 / (peak_m * 1e9)
    out = {"workload": SHORT_WORKLOAD, "prompt_len": P, "resp_len": w.resp_lens[0], "group": G,
           "steps": n, "ms_per_step": round(ms, 3),
           "value": round(sum(replay_flops(P, R, hq, d) for R in w.resp_lens) / (ms * 1e-3) / 1e12, 2),
           "unit": "TFLOP/s", "replays_per_s": round(G / (ms * 1e-3), 2),
           "peaks": {"hbm_gbs": peak_m, "bf16_tflops_sustained": peak_t,
                     "ridge_flop_per_byte": round(ridge, 1)}}
    R = w.resp_lens[0]
    legs = {}
    for name, kern, coef in (("fwd", "tc_fwd", 4.0), ("bwd", "tc_bwd_dq", 6.0)):
        n_l, t_l = trace.get(kern, (0, 0.0))
        if n_l == 0:
            continue
        lms = t_l / n_l
        fl = coef * R * P * d * hq
        gbs = kv / (lms * 1e-3) / 1e9
        intensity = fl / kv
        legs[name] = lms
        out[name] = {"kernel": kern, "launch_ms": round(lms, 3), "prompt_kv_gbs": round(gbs, 1),
                     "hbm_frac": round(gbs / peak_m, 4),
                     "tflops": round(fl / (lms * 1e-3) / 1e12, 1),
                     "tensor_frac": round(fl / (lms * 1e-3) / 1e12 / peak_t, 4),
                     "flop_per_byte": round(intensity, 1),
                     "hbm_frac_ceiling": round(min(1.0, ridge / intensity), 4),
                     "traffic": recorded_traffic(kern, SHORT_WORKLOAD,
                                                 ROOT / "long_context_grpo_replay_gb300" / "csrc" /
                                                 ("ls_tc_fwd.cu" if name == "fwd" else "ls_tc_bwd.cu"))}
    if "fwd" in legs and "bwd" in legs:
        gbs = 2 * kv / ((legs["fwd"] + legs["bwd"]) * 1e-3) / 1e9
        inten = 10.0 * R * P * d * hq / (2 * kv)
        out["fwd_bwd"] = {"prompt_kv_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak_m, 4),
                          "flop_per_byte": round(inten, 1),
                          "hbm_frac_ceiling": round(min(1.0, ridge / inten), 4)}
    out["kernels_ms_per_step"] = {k: round(v[1] / n, 3) for k, v in trace.items()}
    out["target"] = "0.75 of HBM asked; the ceiling above is what the intensity allows"
    del members
    return out


def memory_vs_group(w, desc, prompt, ws, stream, dev):
    """Peak device memory of one group replay at G = 2 and G = 8 (the
    default workload's members: 4096 tokens each) with the prompt pages and
    the workspace resident: the analogue of the pages' 2M-position G=2 vs G=8
    peaks.  The workspace is sized for the longest member, so the two peaks
    should differ by the six extra members' own inputs and outputs alone.
    'non_torch_gib' is device memory in use outside PyTorch's allocator: the
    library allocates nothing, so it must not move with G either."""
    import torch

    import long_context_grpo_replay_gb300.binding as ls
    from long_context_grpo_replay_gb300 import inputs

    res = {}
    io = {}
    for G in (2, 8):
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        members = []
        for g in range(G):
            m = inputs.make_member(w, g, dev)
            R = m["q"].shape[0]
            m.update(o=torch.empty_like(m["q"]),
                     lse=torch.empty(R, w.hq, device=dev, dtype=torch.float32),
                     delta=torch.empty(R, w.hq, device=dev, dtype=torch.float32),
                     dq=torch.empty_like(m["q"]), dk=torch.empty_like(m["k"]),
                     dv=torch.empty_like(m["v"]))
            members.append(m)
        ls.ls_replay_group(desc, prompt, members, ws, stream)
        torch.cuda.synchronize(dev)
        ls.ls_read_device_status(ws)
        free, total = torch.cuda.mem_get_info(dev)
        io[G] = sum(t.numel() * t.element_size() for m in members for t in m.values())
        res[f"G{G}"] = {"peak_allocated_gib": round(torch.cuda.max_memory_allocated(dev) / 2**30, 3),
                        "members_io_gib": round(io[G] / 2**30, 3),
                        "non_torch_gib": round((total - free - torch.cuda.memory_reserved(dev))
                                               / 2**30, 3)}
        del members
    res["peak_delta_gib"] = round(res["G8"]["peak_allocated_gib"] - res["G2"]["peak_allocated_gib"], 3)
    res["extra_members_io_gib"] = round((io[8] - io[2]) / 2**30, 3)
    res["workspace_gib"] = round(ws.numel() / 2**30, 3)
    return res


def run_e2e(args, w, desc, src, members, k_pool, v_pool, pt, prompt, ws, stream, dev, flops_step,
            world):
    """Same step through the public API with pinned host inputs: H2D of the
    prompt K/V, page table and member inputs, the page write and the replay,
    D2H of the outputs.  Like a data loader, the next step's inputs are
    copied on a second stream into a second set of device buffers while this
    step computes, so each step's H2D is inside the timed region but off its
    critical path (the first step's is not hidden)."""
    import torch
    import long_context_grpo_replay_gb300.binding as ls

    in_keys = ("q", "k", "v", "d_o")
    out_keys = ("o", "lse", "dq", "dk", "dv")
    h_src = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in src.items()}
    for k in h_src:
        h_src[k].copy_(src[k])
    h_in = [{k: torch.empty(m[k].shape, dtype=m[k].dtype, pin_memory=True).copy_(m[k])
             for k in in_keys} for m in members]
    h_out = [{k: torch.empty(m[k].shape, dtype=m[k].dtype, pin_memory=True) for k in out_keys}
             for m in members]
    h2d = sum(t.numel() * t.element_size() for t in h_src.values()) + \
        sum(t.numel() * t.element_size() for m in h_in for t in m.values())
    d2h = sum(t.numel() * t.element_size() for m in h_out for t in m.values())

    # two device buffer sets: [0] reuses the bench's tensors, [1] is new
    d_src = [src, {k: torch.empty_like(v) for k, v in src.items()}]
    d_mem = [members, [dict(m, **{k: torch.empty_like(m[k]) for k in in_keys + out_keys})
                       for m in members]]
    # each set's replay reads the page table that set's step copied in
    prompts = [prompt, ls.prompt_from(k_pool, v_pool, d_src[1]["page_table"], w.prompt_len)]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    released = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d_into(b):
        copy_stream.wait_event(released[b])  # the set's previous step is done with it
        with torch.cuda.stream(copy_stream):
            for k in h_src:
                d_src[b][k].copy_(h_src[k], non_blocking=True)
            for m, hm in zip(d_mem[b], h_in):
                for k in in_keys:
                    m[k].copy_(hm[k], non_blocking=True)
        copied[b].record(copy_stream)

    def run(n):
        h2d_into(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                h2d_into(b ^ 1)
            stream.wait_event(copied[b])
            ls.ls_kv_page_write(desc, k_pool, v_pool, d_src[b]["page_table"], 0, d_src[b]["k"],
                                d_src[b]["v"], ws, stream)
            ls.ls_replay_group(desc, prompts[b], d_mem[b], ws, stream)
            with torch.cuda.stream(stream):
                for m, hm in zip(d_mem[b], h_out):
                    for k in out_keys:
                        hm[k].copy_(m[k], non_blocking=True)
            released[b].record(stream)

    for b in (0, 1):
        released[b].record(stream)
    run(1)
    torch.cuda.synchronize()
    n = max(1, args.steps)  # as many steps as the device-timed region: the first H2D is amortised
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    run(n)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / n, dev)
    return {"value": round(job_throughput(flops_step, world, ms), 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": n, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "overlap": "next step's H2D on a copy stream into a second buffer set"}


def _oracle_sample(w, k_pool, v_pool, pt, member, rows, kv=0):
    """Oracle forward+backward of response rows `rows` of the query heads of KV
    head `kv` (a bounded sample of the workload); returns (seconds, flops)."""
    import oracle.ref as ref

    gq = w.hq // w.hkv
    hs = slice(kv * gq, (kv + 1) * gq)
    t0 = time.perf_counter()
    ref.replay_member(k_pool[:, kv:kv + 1], v_pool[:, kv:kv + 1], pt, w.prompt_len,
                      member["q"][:, hs], member["k"][:, kv:kv + 1], member["v"][:, kv:kv + 1],
                      member["d_o"][:, hs], scale=w.scale, rows=rows)
    dt = time.perf_counter() - t0
    d = w.head_dim
    flops = sum(gq * (10.0 * w.prompt_len * d + 14.0 * d * (int(r) + 1)) for r in rows)
    return dt, flops


def cpu_baseline(w, k_pool, v_pool, pt, members, budget_s=20.0):
    import numpy as np
    import torch

    kp = k_pool.cpu()
    vp = v_pool.cpu()
    ptc = pt.cpu()
    m0 = {k: members[0][k].cpu() for k in ("q", "k", "v", "d_o")}
    R = m0["q"].shape[0]
    rows = np.array([R - 1])
    dt, fl = _oracle_sample(w, kp, vp, ptc, m0, rows)
    n_rows = len(rows) * (w.hq // w.hkv)  # query-head rows the sample replays
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"member 0, response row {R - 1} of the {w.hq // w.hkv} query heads of KV "
                      f"head 0, forward+backward over all {w.prompt_len} prompt keys "
                      f"(float64 numpy; {dt:.1f} s)",
            "seconds": round(dt, 2),
            "rows_per_s": round(n_rows / dt, 3),
            # the member's algorithmic flops at the sample's rate
            "extrapolated_s_per_member": round(replay_flops(w.prompt_len, R, w.hq, w.head_dim) / (fl / dt), 1)}


def run_reference(args):
    """The reference arm: the float64 CPU oracle timed on this host, on a
    bounded sample of the same workload per step."""
    import numpy as np
    import torch

    from long_context_grpo_replay_gb300 import inputs

    world, rank, local = dist_env()
    if rank != 0:
        return
    if args.workload in GDN_WORKLOADS:
        return run_reference_gdn(args, world)
    if args.workload in PREFILL_WORKLOADS:
        return run_reference_prefill(args, world)
    w = inputs.WORKLOADS[args.workload]
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    pr = inputs.make_prompt(w, gen_dev)
    kp, vp, pt = pr["k_pool"].cpu(), pr["v_pool"].cpu(), pr["page_table"].cpu()
    m0 = {k: v.cpu() for k, v in inputs.make_member(w, 0, gen_dev).items()}
    del pr
    R = m0["q"].shape[0]
    rows = np.array([R - 1])
    for _ in range(args.warmup):
        _oracle_sample(w, kp, vp, pt, m0, rows)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = _oracle_sample(w, kp, vp, pt, m0, rows)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = (f"per step: member 0, response row {R - 1} of the {w.hq // w.hkv} query heads of "
              f"KV head 0, forward+backward over all {w.prompt_len} prompt keys (float64 numpy)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": replay_config(args.workload, w, world, args.host_pages, args.host_pages_member_major),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _reference_line(args, world, metric, value, unit, dtype, config, sample, ms):
    return {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_gdn(args, world):
    """Oracle arm of a GDN workload: per step the float64 oracle replays the
    first tokens of one head of one member, forward and backward."""
    from long_context_grpo_replay_gb300 import inputs
    from oracle.gdn import gdn_replay

    B, H, R, _ = GDN_WORKLOADS[args.workload]
    n_tok = min(R, 256)
    c = inputs.make_gdn_group(1, 1, n_tok, seed=55)  # same distributions, one (member, head)
    a = {x: t[0] if x != "s0" else t for x, t in c.items()}

    def one():
        t0 = time.perf_counter()
        gdn_replay(a["s0"], a["q"], a["k"], a["v"], a["g"], a["beta"], a["d_o"])
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    tot = sum(one() for _ in range(args.steps))
    value = n_tok * args.steps / H / tot  # whole tokens (all H heads) per second
    line = _reference_line(
        args, world, GDN_METRIC, value, "tokens/s", "f64",
        gdn_config(args.workload, world),
        f"per step: one head of one member, {n_tok} tokens, forward+backward (float64 torch, "
        f"autograd), scaled to {H} heads", tot / args.steps * 1e3)
    print(json.dumps(line), flush=True)


def run_reference_prefill(args, world):
    """Oracle arm of a prefill workload: per step the last prompt row of the
    query heads of one KV head, over all prompt keys."""
    import torch

    import oracle.ref as ref
    from long_context_grpo_replay_gb300 import inputs

    N = PREFILL_WORKLOADS[args.workload]
    w = inputs.Workload(args.workload, 24, 4, 256, 256, N, (N,), "bf16", seed=31)
    gq = w.hq // w.hkv
    hs = inputs.make_head_sample(w, N)
    # The last prompt row sees all N keys: keys 0..N-2 as prompt pages of the
    # one KV head, key N-1 as its own (causal) key, the query as a single row.
    pages = N // w.page_size
    k_pool = hs["k"].view(pages, w.page_size, 1, w.head_dim).transpose(1, 2).contiguous()
    v_pool = hs["v"].view(pages, w.page_size, 1, w.head_dim).transpose(1, 2).contiguous()
    table = torch.arange(pages, dtype=torch.int32)

    def one():
        t0 = time.perf_counter()
        ref.replay_member(k_pool, v_pool, table, N - 1, hs["q"], hs["k"][N - 1:], hs["v"][N - 1:],
                          scale=w.scale)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    tot = sum(one() for _ in range(args.steps))
    value = 4.0 * w.head_dim * gq * N * args.steps / tot / 1e12
    line = _reference_line(
        args, world, PREFILL_METRIC, value, "TFLOP/s", "f64",
        prefill_config(args.workload, world),
        f"per step: row {N - 1} of the {gq} query heads of KV head 0 over all {N} keys "
        "(float64 numpy)", tot / args.steps * 1e3)
    print(json.dumps(line), flush=True)


PREFILL_WORKLOADS = {"prefill_bf16_p32k": 32768, "prefill_bf16_p256k": 262144,
                     "prefill_bf16_p2m": 2097152}
PREFILL_METRIC = "prompt prefill (page write + causal attention) TFLOP/s"


def prefill_config(workload: str, world: int) -> dict:
    """The config object of a prefill line; both arms print the same one."""
    N = PREFILL_WORKLOADS[workload]
    return {"workload": workload, "prompt_len": N, "hq": 24, "hkv": 4, "head_dim": 256,
            "page_size": 256, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (Q %.1f GiB)" % (N * 24 * 256 * 2 / 2**30)}


def prefill_flops(N, hq, d):
    return 4.0 * d * hq * N * (N + 1) / 2.0


def run_prefill(args):
    """The capture step, ls_prompt_prefill: page write of the prompt K/V and
    causal self-attention of the prompt (24/4 heads, d=256, bf16)."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import long_context_grpo_replay_gb300.binding as ls
    from long_context_grpo_replay_gb300 import build, inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    ls.lib()
    N = PREFILL_WORKLOADS[args.workload]
    w = inputs.Workload(args.workload, 24, 4, 256, 256, N, (N,), "bf16", seed=31 + 1000 * rank)
    hq, hkv, d = w.hq, w.hkv, w.head_dim
    desc = ls.desc_for(hq, hkv, d, w.page_size, torch.bfloat16, w.scale)
    pr = inputs.make_prompt(w, dev)
    k_pool, v_pool, pt = pr["k_pool"], pr["v_pool"], pr["page_table"]
    m = inputs.make_member(w, 0, dev, resp_len=N)
    q, k, v = m["q"], m["k"], m["v"]
    del m["d_o"]
    o = torch.empty_like(q)
    lse = torch.empty(N, hq, device=dev, dtype=torch.float32)
    ws = torch.empty(ls.ls_prompt_prefill_workspace_size(desc, N), dtype=torch.uint8, device=dev)
    ls.ls_clear_device_status(ws)
    stream = torch.cuda.current_stream(dev)

    def step(qq, kk, vv):
        ls.ls_prompt_prefill(desc, qq, kk, vv, o, lse, k_pool, v_pool, pt, ws, stream)

    for _ in range(args.warmup):
        step(q, k, v)
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)
    ls.ls_trace_enable(True)
    ls.ls_trace_reset()
    launches0 = ls.ls_launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step(q, k, v)
        e1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = ls.ls_launch_count() - launches0
    trace = ls.kernel_trace()
    ls.ls_trace_enable(False)
    ls.ls_read_device_status(ws)
    clocks = clk.summary()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
    fl = prefill_flops(N, hq, d)
    value = job_throughput(fl, world, ms)

    pk, pk_src = peaks()
    dom = "tc_fwd" if "tc_fwd" in trace else "simt_fwd"
    n_l, t_l = trace.get(dom, (1, ms * args.steps))
    launch_ms = t_l / max(1, n_l)
    peak_t = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = fl / (launch_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
            "frac": achieved / peak_t, "traffic": None, "kernel": dom,
            "peak_source": f"{pk_src} (bf16_tflops_sustained)", "algorithmic_per_launch": fl,
            "launch_ms": launch_ms}

    e2e = None
    if not args.no_e2e:
        hq_, hk_, hv_ = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
                         for t in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        dq_, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def e2e_step():
            dq_.copy_(hq_, non_blocking=True)
            dk_.copy_(hk_, non_blocking=True)
            dv_.copy_(hv_, non_blocking=True)
            step(dq_, dk_, dv_)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n = max(1, min(args.steps, 3))
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(a0.elapsed_time(a1) / n, dev)
        e2e = {"value": round(job_throughput(fl, world, ems), 3), "unit": "TFLOP/s",
               "ms_per_step": round(ems, 3), "steps": n,
               "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))),
               "d2h_bytes_per_step": int(ho.numel() * ho.element_size() + hl.numel() * 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle.ref as ref
        gq = hq // hkv
        qc = q[:, :gq].cpu()
        t0 = time.perf_counter()
        dummy = k_pool[:1, :1].cpu()  # no prompt pages: the prompt is the causal part
        ref.replay_member(dummy, dummy, pt[:1].cpu(), 0, qc, k[:, :1].cpu(), v[:, :1].cpu(),
                          scale=w.scale, rows=np.array([N - 1]))
        dt = time.perf_counter() - t0
        cpu = {"value": 4.0 * d * gq * N / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle",
               "sample": f"row {N - 1} of the {gq} query heads of KV head 0 over all {N} keys "
                         f"(float64 numpy; {dt:.2f} s)", "seconds": round(dt, 2)}

    if rank == 0:
        print(json.dumps({
            "metric": PREFILL_METRIC, "value": round(value, 3), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1)/sqrt(d) Q/K/V, random page table)",
            "config": prefill_config(args.workload, world),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks,
            "kernels_ms_per_step": {kk: round(vv[1] / args.steps, 3) for kk, vv in trace.items()},
        }), flush=True)
    if world > 1:
        dist.destroy_process_group()


# (members, heads, tokens, precision): f32 = the float32 recurrence
# (LS_GDN_EXACT), tc = the chunkwise tensor-core path (LS_GDN_TENSOR_CORE)
GDN_WORKLOADS = {"gdn_f32_h32_r4096_g8": (8, 32, 4096, 0), "gdn_f32_h32_r1024_g4": (4, 32, 1024, 0),
                 "gdn_tc_h32_r4096_g8": (8, 32, 4096, 1), "gdn_tc_h32_r1024_g4": (4, 32, 1024, 1)}
GDN_METRIC = "GDN state replay (forward+backward) response tokens/s per layer"


def fp32_alu_tflops(dev, clocks) -> tuple:
    """fp32 FMA peak of this device: SMs (queried) x 128 lanes x 2 flop x the
    maximum SM clock nvidia-smi reported (2070 MHz when unsampled)."""
    import torch

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_max_mhz") or 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12, sms, mhz

GDN_FWD_FLOP_PER_TOKEN_HEAD = 7   # x dk*dv: S k, the state update, S q
GDN_BWD_FLOP_PER_TOKEN_HEAD = 20  # x dk*dv: S_t, G, G k, S_t^T dO, <G,S>, dk's two products, G decay
GDN_CP_BWD_PRODUCTS = 20  # prep 3, chains 5, outputs 12 (128 x 128 x 128 each, per chunk and head)


def gdn_config(workload: str, world: int) -> dict:
    """The config object of a GDN line; both arms print the same one."""
    B, H, R, prec = GDN_WORKLOADS[workload]
    return {"workload": workload, "group": B, "heads": H, "resp_len": R, "dk": 128, "dv": 128,
            "precision": "LS_GDN_EXACT" if prec == 0 else "LS_GDN_TENSOR_CORE",
            "bwd_reuses_forward": prec != 0,  # LS_GDN_BWD_REUSES_FORWARD: one forward per backward
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (%.1f GiB of q/k/v/dO)" % (4 * B * R * H * 128 * 4 / 2**30)}


def run_gdn(args):
    """Gated-DeltaNet replay of one layer for a group: ls_gdn_replay_fwd (with
    the final state) and ls_gdn_replay_bwd, float32, dk = dv = 128; on the
    tensor-core path the backward reuses the forward's workspace terms."""
    import torch
    import torch.distributed as dist

    import long_context_grpo_replay_gb300.binding as ls
    from long_context_grpo_replay_gb300 import build, inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    ls.lib()
    B, H, R, prec = GDN_WORKLOADS[args.workload]
    D = 128
    c = inputs.make_gdn_group(B, H, R, seed=55 + 1000 * rank, device=dev)
    o = torch.empty_like(c["v"])
    s_final = torch.empty((B, H, D, D), device=dev, dtype=torch.float32)
    gr = {n: torch.empty_like(c[x]) for n, x in
          (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    ws = torch.empty(ls.ls_gdn_workspace_size(ls.GdnDesc(B, H, D, D, prec), R), dtype=torch.uint8,
                     device=dev)
    ls.ls_clear_device_status(ws)
    stream = torch.cuda.current_stream(dev)

    def step(x):
        ls.ls_gdn_replay_fwd(x["s0"], x["q"], x["k"], x["v"], x["g"], x["beta"], o, s_final, ws, stream,
                             precision=prec)
        ls.ls_gdn_replay_bwd(x["s0"], x["q"], x["k"], x["v"], x["g"], x["beta"], x["d_o"],
                             gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], ws, stream,
                             precision=prec, reuse_forward=prec == ls.LS_GDN_TENSOR_CORE)

    for _ in range(args.warmup):
        step(c)
    torch.cuda.synchronize()
    ls.ls_trace_enable(True)
    ls.ls_trace_reset()
    launches0 = ls.ls_launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step(c)
        e1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = ls.ls_launch_count() - launches0
    trace = ls.kernel_trace()
    ls.ls_trace_enable(False)
    clocks = clk.summary()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
    tokens = B * R
    value = tokens * world / (ms * 1e-3)
    unit_flop = D * D * B * R * H
    n_l, t_l = trace.get("gdn_bwd", (1, ms * args.steps))
    launch_ms = t_l / max(1, n_l)
    fl_bwd = GDN_BWD_FLOP_PER_TOKEN_HEAD * unit_flop
    achieved = fl_bwd / (launch_ms * 1e-3) / 1e12
    traffic = recorded_traffic("gdn_bwd", args.workload,
                               ROOT / "long_context_grpo_replay_gb300" / "csrc" / "ls_gdn.cu")
    alu_peak, sms, alu_mhz = fp32_alu_tflops(dev, clocks)
    roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
            "frac": achieved / alu_peak, "traffic": traffic, "kernel": "gdn_bwd",
            "peak_source": f"derived: {sms} SMs (device query) x 128 fp32 lanes x 2 flop x "
                           f"{alu_mhz:.0f} MHz (maximum SM clock)",
            "algorithmic_per_launch": fl_bwd, "launch_ms": launch_ms}
    if prec == 1:
        # tensor-core path: the backward's three kernels execute 20 products of
        # 128 x 128 x 128 per (chunk, head, member); the solves are not counted.
        # Its algorithmic bytes are the backward's own inputs and outputs
        # (q, k, v, dO, g, beta, s0 in; dq, dk, dv, dg, dbeta out, float32).
        # The bound is the one the intensity (flop per algorithmic byte) puts
        # it under against the ridge of the measured peaks, as for attention;
        # the other view is kept beside it.
        nch = -(-R // 128)
        fl_tc = GDN_CP_BWD_PRODUCTS * 2.0 * 128 ** 3 * nch * H * B
        by_tc = (7 * D + 4) * 4.0 * B * R * H + 4.0 * B * H * D * D
        pk, pk_src = peaks()
        peak_t = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        peak_m = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        ach_t = fl_tc / (launch_ms * 1e-3) / 1e12
        ach_m = by_tc / (launch_ms * 1e-3) / 1e9
        tensor = {"bound": "tensor", "achieved": ach_t, "peak": peak_t, "unit": "TFLOP/s",
                  "frac": ach_t / peak_t, "peak_source": f"{pk_src} (bf16_tflops_sustained)",
                  "algorithmic_per_launch": fl_tc, "launch_ms": launch_ms}
        hbm = {"bound": "hbm", "achieved": ach_m, "peak": peak_m, "unit": "GB/s",
               "frac": ach_m / peak_m, "peak_source": f"{pk_src} (hbm_gbs)",
               "algorithmic_per_launch": by_tc, "launch_ms": launch_ms}
        ridge = peak_t * 1e12 / (peak_m * 1e9)
        intensity = fl_tc / by_tc
        roof, other = (tensor, hbm) if intensity >= ridge else (hbm, tensor)
        roof.update({"traffic": recorded_traffic("gdn_bwd", args.workload,
                                                 ROOT / "long_context_grpo_replay_gb300" / "csrc"
                                                 / "ls_gdn_cp.cu"),
                     "kernel": "gdn_bwd (chunk-parallel: prep_grad, chain, out)",
                     "flop_per_byte": round(intensity, 1), "ridge_flop_per_byte": round(ridge, 1)})
        clock_matched(tensor, pk, clocks)
        clock_matched(hbm, pk, clocks)
        roof[other["bound"] + "_view"] = {kk: vv for kk, vv in other.items() if kk != "bound"}

    e2e = None
    if not args.no_e2e:
        names_in = ("s0", "q", "k", "v", "g", "beta", "d_o")
        host = {x: torch.empty(c[x].shape, dtype=torch.float32, pin_memory=True).copy_(c[x])
                for x in names_in}
        dbuf = {x: torch.empty_like(c[x]) for x in names_in}
        outs = [o, s_final] + list(gr.values())
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]

        def e2e_step():
            for x in names_in:
                dbuf[x].copy_(host[x], non_blocking=True)
            step(dbuf)
            for h_, d_ in zip(hout, outs):
                h_.copy_(d_, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n = max(1, args.steps)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(a0.elapsed_time(a1) / n, dev)
        e2e = {"value": round(tokens * world / (ems * 1e-3), 1), "unit": "tokens/s",
               "ms_per_step": round(ems, 3), "steps": n,
               "h2d_bytes_per_step": int(sum(t.numel() * 4 for t in host.values())),
               "d2h_bytes_per_step": int(sum(t.numel() * 4 for t in hout))}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle.gdn import gdn_replay
        n_tok = min(R, 1024)
        a = {x: c[x].cpu() for x in ("s0", "q", "k", "v", "g", "beta", "d_o")}
        t0 = time.perf_counter()
        gdn_replay(a["s0"][:1], a["q"][0, :n_tok, :1], a["k"][0, :n_tok, :1], a["v"][0, :n_tok, :1],
                   a["g"][0, :n_tok, :1], a["beta"][0, :n_tok, :1], a["d_o"][0, :n_tok, :1])
        dt = time.perf_counter() - t0
        cpu = {"value": n_tok / H / dt, "unit": "tokens/s", "cores": torch.get_num_threads(),
               "kind": "oracle",
               "sample": f"member 0, head 0 of {H}, first {n_tok} tokens, forward+backward "
                         f"(float64 torch, autograd; {dt:.2f} s), scaled to all heads",
               "seconds": round(dt, 2)}

    if rank == 0:
        print(json.dumps({
            "metric": GDN_METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if prec == 0 else "bf16 operands, f32 accumulation",
            "data": "synthetic (seeded unit-norm q/k, N(0,1) v, decay in [0.85,1), beta in [0.05,0.95))",
            "config": gdn_config(args.workload, world),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks,
            "kernels_ms_per_step": {kk: round(vv[1] / args.steps, 3) for kk, vv in trace.items()},
        }), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the short-response leg and the G=2/G=8 memory check")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--host-pages-member-major", action="store_true",
                    help="with --host-pages: one member at a time (the prompt streamed once per "
                         "member and pass) instead of chunk-major over the group")
    ap.add_argument("--host-pages", type=int, default=0,
                    help="keep the prompt pages in pinned host memory, streamed in chunks of "
                         "this many pages (0: pages in HBM)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in PREFILL_WORKLOADS:
        run_prefill(args)
    elif args.workload in GDN_WORKLOADS:
        run_gdn(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
