"""Benchmark: fused SDPA forward + backward on one GB300 per rank.

A step is one pass of the whole hot path -- sdpa_fwd then sdpa_bwd through the
C ABI -- over one batch of the varlen THD GQA training workload (8 sequences,
lengths uniform in [512, 4096] from seed 1001, Hq 32, Hkv 8, D 128, bf16,
top-left causal). Inputs are resident in HBM; L2 is flushed (a 256 MiB write)
between timed steps, outside the timed events.

value = TFLOP/s of fwd+bwd under the stated convention (fwd 4*Hq*D*Sq*Sk per
sequence, halved for causal; bwd 2.5x fwd), summed over ranks.
e2e   = the same metric with the inputs copied from pinned host memory and the
outputs (O, LSE, dQ, dK, dV) copied back inside the timed region, every step;
steps are pipelined (the copy in of step s+1 and the copy out of step s-1 run
on their own streams beside the compute of step s, over two device buffer
sets), and the copies of one step timed alone are reported beside it.

--op fwd times the forward alone (the whole path of the forward-only
workloads: asymmetric head dims, where the backward is declined); its
value counts the forward FLOPs only.

--impl reference runs the float64 CPU oracle (the correctness reference) on a
bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s and % of GB300 dense BF16 peak (D128/D512 causal)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- accounting
def seq_lengths(w, inp):
    if w.layout == "thd":
        return np.diff(inp["cu_seqlens_q"]), np.diff(inp["cu_seqlens_kv"])
    return np.full(w.batch, w.seqlen_q), np.full(w.batch, w.seqlen_kv)


def pairs_per_head(w, lq, lk):
    """Exact number of unmasked (query, key) pairs of one head, one sequence."""
    i = np.arange(lq, dtype=np.int64)
    off = lk - lq if w.mask == "causal_br" else 0
    wl, wr = w.window
    if w.mask != "none":
        wr = 0
    lo = np.maximum(0, i + off - wl) if wl >= 0 else np.zeros_like(i)
    hi = np.minimum(lk, np.maximum(0, i + off + wr + 1)) if wr >= 0 else np.full_like(i, lk)
    return int(np.maximum(0, hi - lo).sum())


def flops(w, inp):
    """(fwd_convention, fwd_exact) FLOPs of one forward over the workload:
    2*D (Q K^T) + 2*Dv (P V) per (query, key) pair per head, i.e. 4*D for
    equal head dims."""
    lqs, lks = seq_lengths(w, inp)
    per_pair = 2 * w.head_dim + 2 * w.dv
    conv = exact = 0
    for lq, lk in zip(lqs, lks):
        c = per_pair * w.heads_q * int(lq) * int(lk)
        conv += c // 2 if w.mask != "none" else c
        exact += per_pair * w.heads_q * pairs_per_head(w, int(lq), int(lk))
    return conv, exact


def forward_only(args, w):
    return args.op == "fwd" or w.name in workloads.FORWARD_ONLY


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- oracle arm
_sample_cache = {}


def sample_arrays(w, inp, ls, nkv=1, fwd_only=False):
    """The first `ls` query tokens of sequence 0 (and the keys they can see
    under the workload's alignment), `nkv` kv heads with their q heads,
    rounded to the workload dtype."""
    key = (w.name, ls, nkv, fwd_only)
    if key in _sample_cache:
        return _sample_cache[key]
    rin = workloads.rounded(inp, w.dtype)
    group = w.heads_q // w.heads_kv * nkv
    if w.layout == "thd":
        lq0 = int(inp["cu_seqlens_q"][1] - inp["cu_seqlens_q"][0])
        lk0 = int(inp["cu_seqlens_kv"][1] - inp["cu_seqlens_kv"][0])
    else:
        lq0, lk0 = w.seqlen_q, w.seqlen_kv
    lq = min(ls, lq0)
    lk = min(lk0, lq + (lk0 - lq0)) if w.mask == "causal_br" else min(lk0, lq) if lq0 == lk0 else lk0
    if w.layout == "thd":
        q0, k0 = int(inp["cu_seqlens_q"][0]), int(inp["cu_seqlens_kv"][0])
        q, do = (rin[x][q0:q0 + lq, :group] for x in ("q", "do"))
        k, v = (rin[x][k0:k0 + lk, :nkv] for x in ("k", "v"))
        kw = dict(layout="thd", cu_q=np.array([0, lq], np.int32), cu_kv=np.array([0, lk], np.int32))
    elif w.layout == "bshd":
        q, do = (rin[x][:1, :lq, :group] for x in ("q", "do"))
        k, v = (rin[x][:1, :lk, :nkv] for x in ("k", "v"))
        kw = dict(layout="bshd")
    else:
        q, do = (rin[x][:lq, :1, :group] for x in ("q", "do"))
        k, v = (rin[x][:lk, :1, :nkv] for x in ("k", "v"))
        kw = dict(layout="sbhd")
    arrs = tuple(np.ascontiguousarray(a) for a in (q, k, v, do))
    sub = w.replace(layout="bshd", batch=1, seqlen_q=lq, seqlen_kv=lk, heads_q=group, heads_kv=nkv)
    conv, _ = flops(sub, {})
    out = (arrs, kw, conv if fwd_only else 3.5 * conv, lq, group)
    _sample_cache[key] = out
    return out


def time_oracle(w, inp, ls, nkv=1, fwd_only=False):
    from oracle import oracle

    (q, k, v, do), kw, fl, lq, group = sample_arrays(w, inp, ls, nkv, fwd_only)
    t0 = time.perf_counter()
    if fwd_only:
        oracle.fwd(q, k, v, mask=w.mask, scale=w.scale, window=w.window, **kw)
    else:
        oracle.bwd(q, k, v, do, mask=w.mask, scale=w.scale, window=w.window, **kw)
    return time.perf_counter() - t0, fl, lq, group


def oracle_sample(w, inp, seconds_target: float, fwd_only=False):
    """Grow the sample until one float64 oracle fwd+bwd (or fwd) takes about `seconds_target`."""
    from oracle import oracle

    ls, nkv = 256, 1
    dt, fl, lq, group = time_oracle(w, inp, ls, nkv, fwd_only)
    while dt < seconds_target * 0.6 and lq == ls:
        ls = int(ls * min(2.0, max(1.15, (seconds_target / max(dt, 1e-3)) ** 0.5)))
        dt, fl, lq, group = time_oracle(w, inp, ls, nkv, fwd_only)
    while dt < seconds_target * 0.6 and nkv < w.heads_kv:
        nkv = min(w.heads_kv, max(nkv + 1, int(nkv * seconds_target / max(dt, 1e-3))))
        dt, fl, lq, group = time_oracle(w, inp, ls, nkv, fwd_only)
    return {"seconds": dt, "flops": fl, "tflops": fl / dt / 1e12, "ls": lq, "group": group, "nkv": nkv,
            "threads": oracle.num_threads()}


def reference_arm(args, w, inp):
    if rank_env()[1] != 0:  # the CPU baseline runs once, on rank 0
        return
    fo = forward_only(args, w)
    per_step = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    s = oracle_sample(w, inp, per_step, fo)
    times = []
    for it in range(args.warmup + args.steps):
        dt, fl, _, _ = time_oracle(w, inp, s["ls"], s["nkv"], fo)
        if it >= args.warmup:
            times.append(dt)
    t = float(np.mean(times))
    value = s["flops"] / t / 1e12
    sample = (f"float64 oracle {'fwd' if fo else 'fwd+bwd'} of the first {s['ls']} query tokens of sequence 0 "
              f"with {s['nkv']} kv head(s) ({s['group']} q heads), per step")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": s["threads"], "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ranks
def rank_env():
    """(world, rank, local_rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank timings: the slowest rank sets the job's time."""
    import torch

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_tflops(world, flops_per_step, steps, ms):
    """Whole-job TFLOP/s: every rank runs the same workload (replicas, weak
    scaling), so the job does world x the work of one rank in the slowest
    rank's time."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- GPU arm
def gpu_arm(args, w, inp):
    import torch
    import torch.distributed as dist

    import scaled_dot_product_02_gb300 as sdpa

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    dev = torch.device("cuda", local)
    fo = forward_only(args, w)
    ins = ("q", "k", "v") if fo else ("q", "k", "v", "do")
    outs = ("o", "lse") if fo else ("o", "lse", "dq", "dk", "dv")
    host = {x: workloads.to_torch(inp[x], w.dtype).pin_memory() for x in ins}
    q, k, v = (host[x].to(dev) for x in ("q", "k", "v"))
    do = None if fo else host["do"].to(dev)
    kw = dict(layout=w.layout, mask=w.mask, scale=w.scale, window=w.window)
    host_cu = {}
    if w.layout == "thd":
        for x in ("cu_seqlens_q", "cu_seqlens_kv"):
            host_cu[x] = torch.from_numpy(inp[x]).pin_memory()
        kw.update(cu_seqlens_q=host_cu["cu_seqlens_q"].to(dev), cu_seqlens_kv=host_cu["cu_seqlens_kv"].to(dev),
                  max_seqlen_q=int(np.max(np.diff(inp["cu_seqlens_q"]))),
                  max_seqlen_kv=int(np.max(np.diff(inp["cu_seqlens_kv"]))))
    o = torch.empty(tuple(q.shape[:-1]) + (w.dv,), dtype=q.dtype, device=dev)
    rows_q = q.numel() // (w.heads_q * w.head_dim)
    lse = torch.empty((rows_q, w.heads_q), dtype=torch.float32, device=dev)
    batch = len(inp["cu_seqlens_q"]) - 1 if w.layout == "thd" else None
    prob = sdpa.make_problem(q, k, layout=w.layout, mask=w.mask, window=w.window, scale=w.scale, batch=batch,
                             max_seqlen_q=kw.get("max_seqlen_q"), max_seqlen_kv=kw.get("max_seqlen_kv"),
                             head_dim_v=w.dv, kv_chunk=args.kv_chunk)
    ws_f = torch.empty(max(256, sdpa.sdpa_fwd_workspace_size(prob)), dtype=torch.uint8, device=dev)
    dq = dk = dv = ws_b = None
    if not fo:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws_b = torch.empty(max(256, sdpa.sdpa_bwd_workspace_size(prob)), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    det = bool(args.deterministic)

    def step():
        sdpa.sdpa_fwd(q, k, v, out=o, lse=lse, workspace=ws_f, **kw)
        n = sdpa.sdpa_last_launch_count()
        if fo:
            return n
        sdpa.sdpa_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws_b, deterministic=det,
                      kv_chunk=args.kv_chunk, **kw)
        return n + sdpa.sdpa_last_launch_count()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sdpa.sdpa_profile_begin()
    launches = 0
    for i in range(args.steps):
        flush.fill_(i & 255)
        starts[i].record()
        launches += step()
        ends[i].record()
    torch.cuda.synchronize()
    prof = sdpa.sdpa_profile_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during the timed steps")

    # end to end: host buffers in, results back out, every step. Steps are
    # pipelined over two device buffer sets and three streams: the host->device
    # copy of step s+1 and the device->host copy of step s-1 run beside the
    # compute of step s (the link is full duplex). Every step still copies its
    # own inputs in and its own results out inside the timed region.
    dev_out = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    h_out = {x: torch.empty(dev_out[x].shape, dtype=dev_out[x].dtype, pin_memory=True) for x in outs}
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + sum(
        t.numel() * t.element_size() for t in host_cu.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    e_steps = max(2, args.steps // 2)
    sets = []
    for b in range(2):
        dset = {x: torch.empty_like(t) for x, t in (("q", q), ("k", k), ("v", v), ("do", do), ("o", o), ("lse", lse),
                                                     ("dq", dq), ("dk", dk), ("dv", dv), ("ws_f", ws_f), ("ws_b", ws_b))
                if t is not None}
        for x in host_cu:
            dset[x] = torch.empty_like(kw[x])
        sets.append(dset)
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])  # step i-2 has finished reading this set's inputs
            for x in ins:
                d[x].copy_(host[x], non_blocking=True)
            for x in host_cu:
                d[x].copy_(host_cu[x], non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        if i >= 2:
            s_comp.wait_event(ev_out[b])  # step i-2's results have left this set
        kwb = dict(kw)
        for x in host_cu:
            kwb[x] = d[x]
        sdpa.sdpa_fwd(d["q"], d["k"], d["v"], out=d["o"], lse=d["lse"], workspace=d["ws_f"], stream=s_comp, **kwb)
        if not fo:
            sdpa.sdpa_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], dq=d["dq"], dk=d["dk"], dv=d["dv"],
                          workspace=d["ws_b"], stream=s_comp, deterministic=det, kv_chunk=args.kv_chunk, **kwb)
        ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for x in outs:
                h_out[x].copy_(d[x], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error in the end-to-end warm-up")
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e_steps):
        e2e_step(i)
    s_comp.wait_stream(s_in)
    s_comp.wait_stream(s_out)
    e1.record(s_comp)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during the end-to-end steps")
    # the copies of a step, each timed alone (context for the overlap)
    ta, tb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ta.record()
    for x in ins:
        sets[0][x].copy_(host[x], non_blocking=True)
    tb.record()
    torch.cuda.synchronize()
    h2d_ms = ta.elapsed_time(tb)
    ta.record()
    for x in outs:
        h_out[x].copy_(sets[0][x], non_blocking=True)
    tb.record()
    torch.cuda.synchronize()
    d2h_ms = ta.elapsed_time(tb)

    conv, exact = flops(w, inp)
    step_flops = conv if fo else 3.5 * conv
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world, device=dev)
    value = job_tflops(world, step_flops, args.steps, ms)
    e2e_value = job_tflops(world, step_flops, 1, e2e_ms)

    pk, pk_kind = peaks()
    sustained = ms > 1000.0
    peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    if w.dtype == "fp16":
        peak = peak * 1.0  # dense fp16 and bf16 tensor rates are equal on this part
    kern = {}
    for kind in ("fwd", "bwd", "preprocess", "dq_finalize", "guard", "bwd_dq"):
        tot, n = prof[kind]
        kern[kind] = {"ms_total": tot, "launches": n, "ms_avg": tot / n if n else None}
    fwd_alg = exact            # 2*D + 2*Dv (4*D) flop per unmasked pair per head
    bwd_alg = 2.5 * exact      # 10*D flop per unmasked pair per head
    # algorithmic flops per launch of each kernel: the deterministic backward
    # splits the 10*D into the dK/dV kernel (8*D: S, dP, dV, dK) and the dQ
    # pass (2*D of useful work; it also recomputes S and dP)
    alg_of = {"fwd": fwd_alg, "bwd": (2.0 if kern["bwd_dq"]["launches"] else 2.5) * exact, "bwd_dq": 0.5 * exact}
    dom = max((x for x in ("fwd", "bwd", "bwd_dq") if kern[x]["launches"]), key=lambda x: kern[x]["ms_total"])
    alg = alg_of[dom]
    achieved = alg / (kern[dom]["ms_avg"] * 1e-3) / 1e12
    kname = {"fwd": "fwd_kernel", "bwd": "bwd_kernel", "bwd_dq": "dq128_kernel"}[dom]
    roofline = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic_for(dom, w.name) if dom != "bwd_dq" and not args.deterministic else None,
                "peak_source": f"{pk_kind} {'bf16_tflops_sustained' if sustained else 'bf16_tflops'}",
                "algorithmic_flops_per_launch": alg}
    bwd_ms = (kern["bwd"]["ms_total"] + kern["bwd_dq"]["ms_total"]) / args.steps  # whole backward, per step
    detail = {
        "fwd_kernel_tflops_exact": fwd_alg / (kern["fwd"]["ms_avg"] * 1e-3) / 1e12,
        "bwd_kernel_tflops_exact": bwd_alg / (bwd_ms * 1e-3) / 1e12 if not fo else None,
        "fwd_kernel_tflops_convention": conv / (kern["fwd"]["ms_avg"] * 1e-3) / 1e12,
        "bwd_kernel_tflops_convention": 2.5 * conv / (bwd_ms * 1e-3) / 1e12 if not fo else None,
        "step_tflops_exact": world * (1.0 if fo else 3.5) * exact * args.steps / (ms * 1e-3) / 1e12,
        "pct_of_peak_step": 100.0 * value / world / peak,
        "kernels": kern,
        "preprocess_gbs": None,
    }
    if kern["preprocess"]["ms_avg"]:
        # reads O and dO (2 bytes each), writes delta and LSE*log2e, zeroes the fp32 dQ accumulator
        rows = rows_q * w.heads_q
        zeroed = rows * w.head_dim * 4 if kern["dq_finalize"]["launches"] else 0  # fp32 dQ accumulator
        byts = rows * w.head_dim * 2 * 2 + rows * 8 + zeroed
        detail["preprocess_gbs"] = byts / (kern["preprocess"]["ms_avg"] * 1e-3) / 1e9
    if kern["dq_finalize"]["ms_avg"]:
        rows = rows_q * w.heads_q
        detail["dq_finalize_gbs"] = rows * w.head_dim * 6 / (kern["dq_finalize"]["ms_avg"] * 1e-3) / 1e9

    if w.name == workloads.VARLEN_THD.name and not fo and not args.no_companion:
        # the other half of the headline metric (head_dim 512), same process and timing
        detail["d512"] = companion_measure(workloads.D512_BR, max(10, args.steps // 10), args.warmup, dev, flush,
                                           peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(w, inp, 12.0, fo)
        cpu = {"value": s["tflops"], "unit": "TFLOP/s", "cores": s["threads"], "kind": "oracle",
               "sample": f"float64 oracle {'fwd' if fo else 'fwd+bwd'} of the first {s['ls']} query tokens of "
                         f"sequence 0 with {s['nkv']} kv head(s) ({s['group']} q heads): {s['seconds']:.1f} s"}
    lq, _ = seq_lengths(w, inp)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "layout": w.layout, "mask": w.mask, "batch": len(lq),
                       "seq_lengths": [int(x) for x in lq], "heads_q": w.heads_q, "heads_kv": w.heads_kv,
                       "head_dim": w.head_dim, "head_dim_v": w.dv, "window": list(w.window),
                       "pass": "forward only" if fo else "forward + backward",
                       "flop_convention": "fwd (2*D + 2*Dv)*Hq*Sq*Sk per sequence (4*Hq*D*Sq*Sk for equal dims), "
                                          "halved for causal; bwd 2.5x fwd",
                       "l2": "flushed between timed steps (256 MiB write, outside the events)",
                       "parallelism": f"replicas x{world} (no collective)",
                       "backward": None if fo else "deterministic" if det else "fp32 reductions for dQ (head_dim 128)",
                       "bwd_workspace_bytes": None if fo else int(ws_b.numel()),
                       "kv_chunk": None if fo or w.head_dim == 128 else args.kv_chunk or "library choice"},
            "clocks": clk, "gpu_launches": launches,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "h2d_ms_alone": h2d_ms, "d2h_ms_alone": d2h_ms,
                    "overlap": "H2D of step s+1 and D2H of step s-1 beside the compute of step s (3 streams, "
                               "2 device buffer sets)"},
            "roofline": roofline, "cpu_baseline": cpu, "detail": detail}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def merge_arm(args, w, inp):
    """The log-sum-exp merge of key-split partial results (sdpa_merge) over the
    workload's query rows: n_parts blocks of bf16 partial outputs and fp32
    LSE, memory-bound. Prints its own JSON line (GB/s against the measured
    HBM copy bandwidth)."""
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rows = int(np.sum(seq_lengths(w, inp)[0]))
    n_parts, d, heads = args.merge_parts, w.head_dim, w.heads_q
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    po = torch.randn((n_parts, rows, heads, d), device=dev, generator=g).to(torch.bfloat16)
    pl = torch.randn((n_parts, rows, heads), device=dev, generator=g) * 2.0 + 8.0
    pl[0, ::7] = float("-inf")  # blocks without keys for some rows
    o = torch.empty((rows, heads, d), device=dev, dtype=torch.bfloat16)
    lse = torch.empty((rows, heads), device=dev, dtype=torch.float32)
    items = rows * heads
    # algorithmic bytes: every statistic, the rows of non-empty blocks, the outputs
    n_empty = int(torch.isneginf(pl).sum().item())
    nbytes = n_parts * items * 4 + (n_parts * items - n_empty) * d * 2 + items * (d * 2 + 4)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        sdpa.sdpa_merge(po, pl, out=o, lse=lse)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.steps):
        flush.fill_(i & 255)
        starts[i].record()
        sdpa.sdpa_merge(po, pl, out=o, lse=lse)
        ends[i].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during the merge")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    (ms,) = max_over_ranks([ms], world, device=dev)
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk, pk_kind = peaks()
    line = {"metric": "LSE merge of key-split partial results, GB/s", "value": world * gbs, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"lse_merge_{w.name}", "n_parts": n_parts, "items": items, "head_dim": d,
                       "bytes_per_launch": nbytes, "l2": "flushed between timed launches (256 MiB write)"},
            "clocks": clk, "gpu_launches": args.steps,
            "roofline": {"bound": "hbm", "kernel": "merge_kernel", "achieved": gbs, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / pk["hbm_gbs"], "traffic": None,
                         "peak_source": f"{pk_kind} hbm_gbs"}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def companion_measure(w, steps, warmup, dev, flush, peak):
    """Forward and backward of a second workload, timed in the same process
    the same way (CUDA events around each step, L2 flushed between steps,
    per-kernel events from the library's profiler): the headline metric
    names head_dim 128 and 512, and the default step is the head_dim 128
    one. Exact-mask FLOPs (4*D per unmasked pair forward, 10*D backward)."""
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    inp = workloads.make_inputs(w)
    q, k, v, do = (workloads.to_torch(inp[x], w.dtype).to(dev) for x in ("q", "k", "v", "do"))
    kw = dict(layout=w.layout, mask=w.mask, scale=w.scale, window=w.window)
    o = torch.empty_like(q)
    lse = torch.empty((q.numel() // (w.heads_q * w.head_dim), w.heads_q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    prob = sdpa.make_problem(q, k, layout=w.layout, mask=w.mask, window=w.window, scale=w.scale)
    ws_f = torch.empty(max(256, sdpa.sdpa_fwd_workspace_size(prob)), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(256, sdpa.sdpa_bwd_workspace_size(prob)), dtype=torch.uint8, device=dev)

    def step():
        sdpa.sdpa_fwd(q, k, v, out=o, lse=lse, workspace=ws_f, **kw)
        n = sdpa.sdpa_last_launch_count()
        sdpa.sdpa_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws_b, **kw)
        return n, sdpa.sdpa_last_launch_count()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError(f"device error during the {w.name} warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    sdpa.sdpa_profile_begin()
    launches = (0, 0)
    for i in range(steps):
        flush.fill_(i & 255)
        starts[i].record()
        launches = step()
        ends[i].record()
    torch.cuda.synchronize()
    prof = sdpa.sdpa_profile_end()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError(f"device error during the {w.name} steps")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
    conv, exact = flops(w, inp)
    fwd_ms = prof["fwd"][0] / steps
    bwd_ms = sum(prof[x][0] for x in ("preprocess", "bwd", "dq_finalize")) / steps
    out = {"workload": w.name, "steps": steps, "ms_per_step": ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
           "fwd_launches_per_step": launches[0], "bwd_launches_per_step": launches[1],
           "fwd_tflops_exact": exact / (fwd_ms * 1e-3) / 1e12,
           "bwd_tflops_exact": 2.5 * exact / (bwd_ms * 1e-3) / 1e12,
           "fwd_tflops_convention": conv / (fwd_ms * 1e-3) / 1e12,
           "bwd_tflops_convention": 2.5 * conv / (bwd_ms * 1e-3) / 1e12,
           "step_tflops_convention": 3.5 * conv / (ms * 1e-3) / 1e12,
           "peak": peak,
           "bwd_workspace_bytes": int(ws_b.numel()),
           "note": "bwd_ms covers every kernel of the backward call (preprocess, score, GEMMs, dQ finalise)"}
    out["fwd_frac_of_peak"] = out["fwd_tflops_exact"] / peak
    out["bwd_frac_of_peak"] = out["bwd_tflops_exact"] / peak
    del q, k, v, do, o, lse, dq, dk, dv, ws_f, ws_b
    torch.cuda.empty_cache()
    return out


def fp8_oracle_sample(w, inp8, seconds_target):
    """The float64 FP8 oracle on the first query tokens of sequence 0 with one
    kv head and its q heads, grown until one run takes about
    `seconds_target`; returns its TFLOP/s under the exact-mask count."""
    import time

    from oracle import oracle

    group = w.heads_q // w.heads_kv
    lq0 = int(inp8["cu_seqlens_q"][1]) if w.layout == "thd" else w.seqlen_q
    ls, dt, fl = 128, 0.0, 0
    while True:
        lq = min(ls, lq0)
        if w.layout == "thd":
            q8, k8, v8 = inp8["q8"][:lq, :group], inp8["k8"][:lq, :1], inp8["v8"][:lq, :1]
            kw = dict(layout="thd", cu_q=np.array([0, lq], np.int32), cu_kv=np.array([0, lq], np.int32))
        elif w.layout == "bshd":
            q8, k8, v8 = inp8["q8"][:1, :lq, :group], inp8["k8"][:1, :lq, :1], inp8["v8"][:1, :lq, :1]
            kw = dict(layout="bshd")
        else:
            q8, k8, v8 = inp8["q8"][:lq, :1, :group], inp8["k8"][:lq, :1, :1], inp8["v8"][:lq, :1, :1]
            kw = dict(layout="sbhd")
        q8, k8, v8 = (np.ascontiguousarray(x) for x in (q8, k8, v8))
        t0 = time.perf_counter()
        oracle.fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, mask=w.mask, scale=w.scale, window=w.window, **kw)
        dt = time.perf_counter() - t0
        sub = w.replace(layout="bshd", batch=1, seqlen_q=lq, seqlen_kv=lq, heads_q=group, heads_kv=1)
        _, fl = flops(sub, {})
        if dt >= seconds_target * 0.6 or lq == lq0:
            break
        ls = int(ls * min(2.0, max(1.15, (seconds_target / max(dt, 1e-3)) ** 0.5)))
    return {"seconds": dt, "tflops": fl / dt / 1e12, "ls": lq, "group": group, "threads": oracle.num_threads()}


def fp8_arm(args, w, inp):
    """FP8 E4M3 forward (sdpa_fwd_fp8) on the workload's shape with seeded E4M3
    inputs: TFLOP/s under the exact-mask count (4*D per unmasked pair; the
    kernel executes 6*D, S twice), roofline against the dense FP8 peak taken as
    twice the measured bf16 figure (the nominal 4.5 / 2.25 PFLOP/s ratio)."""
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    if w.head_dim not in (128, 256) or w.dv != w.head_dim:
        raise SystemExit("--op fp8 needs a head_dim 128 or 256 workload")
    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp8 = workloads.fp8_inputs(w)
    host = {x: torch.from_numpy(inp8[x]).pin_memory() for x in ("q8", "k8", "v8")}
    q8, k8, v8 = (host[x].to(dev) for x in ("q8", "k8", "v8"))
    kw = dict(layout=w.layout, mask=w.mask, scale=w.scale, window=w.window)
    host_cu = {}
    if w.layout == "thd":
        for x in ("cu_seqlens_q", "cu_seqlens_kv"):
            host_cu[x] = torch.from_numpy(inp8[x]).pin_memory()
        kw.update(cu_seqlens_q=host_cu["cu_seqlens_q"].to(dev), cu_seqlens_kv=host_cu["cu_seqlens_kv"].to(dev),
                  max_seqlen_q=int(np.max(np.diff(inp8["cu_seqlens_q"]))),
                  max_seqlen_kv=int(np.max(np.diff(inp8["cu_seqlens_kv"]))))
    o = torch.empty(tuple(q8.shape), dtype=torch.bfloat16, device=dev)
    rows_q = q8.numel() // (w.heads_q * w.head_dim)
    lse = torch.empty((rows_q, w.heads_q), dtype=torch.float32, device=dev)
    batch = len(inp8["cu_seqlens_q"]) - 1 if w.layout == "thd" else None
    prob = sdpa.make_problem(q8, k8, layout=w.layout, mask=w.mask, window=w.window, scale=w.scale, batch=batch,
                             dtype=0, max_seqlen_q=kw.get("max_seqlen_q"), max_seqlen_kv=kw.get("max_seqlen_kv"))
    ws = torch.empty(max(256, sdpa.sdpa_fwd_fp8_workspace_size(prob)), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        sdpa.sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, out=o, lse=lse, workspace=ws, **kw)
        return sdpa.sdpa_last_launch_count()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    sdpa.sdpa_profile_begin()
    launches = 0
    for i in range(args.steps):
        flush.fill_(i & 255)
        starts[i].record()
        launches += step()
        ends[i].record()
    torch.cuda.synchronize()
    prof = sdpa.sdpa_profile_end()
    clk = clocks.stop()
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during the timed steps")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
    # end to end through the same call: E4M3 inputs in from pinned host memory,
    # O and LSE out, every step, serialised
    h_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    h_l = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h2d = sum(t.numel() for t in host.values()) + sum(t.numel() * 4 for t in host_cu.values())
    d2h = h_o.numel() * 2 + h_l.numel() * 4
    e_steps = max(2, args.steps // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e_steps):
        for x, t in (("q8", q8), ("k8", k8), ("v8", v8)):
            t.copy_(host[x], non_blocking=True)
        for x in host_cu:
            kw[x].copy_(host_cu[x], non_blocking=True)
        step()
        h_o.copy_(o, non_blocking=True)
        h_l.copy_(lse, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    if sdpa.sdpa_get_device_error() != 0:
        raise RuntimeError("device error during the end-to-end steps")
    conv, exact = flops(w, inp)
    value = job_tflops(world, exact, args.steps, ms)
    pk, pk_kind = peaks()
    peak = 2.0 * pk["bf16_tflops"]
    kern_ms = prof["fwd"][0] / max(prof["fwd"][1], 1)
    achieved = exact / (kern_ms * 1e-3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = fp8_oracle_sample(w, inp8, 12.0)
        cpu = {"value": s["tflops"], "unit": "TFLOP/s", "cores": s["threads"], "kind": "oracle",
               "sample": f"float64 FP8 oracle forward of the first {s['ls']} query tokens of sequence 0 with one "
                         f"kv head ({s['group']} q heads): {s['seconds']:.1f} s"}
    line = {"metric": "FP8 E4M3 attention forward TFLOP/s (exact-mask 4*D per unmasked pair)", "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (fp32 accumulate, bf16 O)", "data": "synthetic",
            "config": {"workload": f"{w.name}_fp8", "layout": w.layout, "mask": w.mask, "heads_q": w.heads_q,
                       "heads_kv": w.heads_kv, "head_dim": w.head_dim, "descale": list(workloads.FP8_DESCALE),
                       "inputs": "E4M3 codes of the workload's seeded N(0,1) masters times 3",
                       "l2": "flushed between timed steps (256 MiB write, outside the events)",
                       "parallelism": f"replicas x{world} (no collective)"},
            "clocks": clk, "gpu_launches": launches,
            "e2e": {"value": job_tflops(world, exact, 1, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": "none (serial copies)"},
            "roofline": {"bound": "tensor", "kernel": "fwd_fp8_kernel", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic_for("fwd_fp8", w.name),
                         "peak_source": f"{pk_kind} bf16_tflops x 2 (nominal dense fp8/bf16 ratio 4.5/2.25)",
                         "algorithmic_flops_per_launch": exact, "executed_flops_per_launch": 1.5 * exact},
            "cpu_baseline": cpu,
            "detail": {"kernels_ms_per_step": {k: prof[k][0] / args.steps for k in ("guard", "v_transpose", "fwd")},
                       "fwd_fp8_kernel_tflops_executed": 1.5 * achieved}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def traffic_for(kind, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"traffic_{kind}_kernel_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line:
            a, b = line.split(":", 1)
            vals[a.strip()] = b.strip()
    src = os.path.join(ROOT, "scaled_dot_product_02_gb300", "csrc", f"{kind}.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if vals.get("source_sha256_16") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="varlen_thd_gqa", choices=[w.name for w in workloads.ALL])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="step", choices=["step", "fwd", "merge", "fp8"],
                    help="step: the fwd+bwd hot path (the headline; the forward alone for forward-only "
                         "workloads); fwd: the forward alone; merge: the LSE merge of key-split results; "
                         "fp8: the FP8 E4M3 forward (head_dim 128 or 256 workloads)")
    ap.add_argument("--merge-parts", type=int, default=4)
    ap.add_argument("--kv-chunk", type=int, default=0,
                    help="head_dim 256/512 backward: key positions per chunk (multiple of 128; 0 = library choice)")
    ap.add_argument("--no-companion", action="store_true",
                    help="skip timing the head_dim 512 workload beside the default head_dim 128 step")
    ap.add_argument("--deterministic", action="store_true",
                    help="bitwise-reproducible backward (head_dim 128: separate dQ pass, no fp32 reductions)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = {x.name: x for x in workloads.ALL}[args.workload]
    inp = workloads.make_inputs(w)
    if args.op == "merge":
        merge_arm(args, w, inp)
    elif args.op == "fp8" and args.impl == "ours":
        fp8_arm(args, w, inp)
    elif args.impl == "reference":
        reference_arm(args, w, inp)
    else:
        gpu_arm(args, w, inp)


if __name__ == "__main__":
    main()
