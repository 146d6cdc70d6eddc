"""Parity helpers: run the CUDA path and the float64 oracle on the same seeded
inputs and apply the acceptance rule.

Rule (TransformerEngine PR #3527, "Verification": the criterion FlashAttention
applies to itself, err(kernel, fp64) <= 2 * err(inputs rounded to dtype, fp64),
with the floor measured per case), read as:
  R      = oracle on the float64 master inputs
  floor  = max |round_to_dtype(oracle on dtype-rounded inputs) - R|  per tensor
           (the best a kernel with dtype inputs and dtype outputs could do;
           LSE is float32, so it is not rounded)
  pass   iff max |kernel - R| <= 2 * floor, per tensor,
plus the absolute caps against the oracle on the rounded inputs:
  max |O - O_ref| <= 2e-2 (bf16) / 4e-3 (fp16),  max |LSE - LSE_ref| <= 1e-3.
Rows with no allowed key must be exactly O = 0, LSE = -inf (and dQ = 0).
"""
from __future__ import annotations

import numpy as np

import workloads
from oracle import oracle

O_CAP = {"bf16": 2e-2, "fp16": 4e-3}
LSE_CAP = 1e-3


def torch_dtype(name):
    import torch

    return {"bf16": torch.bfloat16, "fp16": torch.float16}[name]


def to_device(x: np.ndarray, dtype: str):
    return workloads.to_torch(x, dtype).cuda().contiguous()


def oracle_kwargs(w: workloads.Workload, inp):
    kw = dict(layout=w.layout, mask=w.mask, scale=w.scale, window=w.window)
    if w.layout == "thd":
        kw.update(cu_q=inp["cu_seqlens_q"], cu_kv=inp["cu_seqlens_kv"])
    return kw


def gpu_kwargs(w: workloads.Workload, inp):
    import torch

    kw = dict(layout=w.layout, mask=w.mask, scale=w.scale, window=w.window)
    if w.layout == "thd":
        cq, ck = inp["cu_seqlens_q"], inp["cu_seqlens_kv"]
        kw.update(cu_seqlens_q=torch.from_numpy(cq).cuda(), cu_seqlens_kv=torch.from_numpy(ck).cuda(),
                  max_seqlen_q=int(np.max(np.diff(cq))) if len(cq) > 1 else 0,
                  max_seqlen_kv=int(np.max(np.diff(ck))) if len(ck) > 1 else 0)
    return kw


def max_abs(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nanmax(d)) if d.size else 0.0


def judge(name, got, ref_master, ref_rounded, dtype, cap=None, round_out=True):
    """Returns (ok, message) for one tensor."""
    floor_src = workloads.round_to(ref_rounded, dtype) if round_out else ref_rounded
    floor = max_abs(floor_src, ref_master)
    err = max_abs(got, ref_master)
    err_r = max_abs(got, ref_rounded)
    ok = err <= 2.0 * floor + 1e-12 and np.all(np.isfinite(got) | np.isinf(ref_rounded))
    if cap is not None:
        ok = ok and err_r <= cap
    return ok, f"{name}: err={err:.3e} floor={floor:.3e} ratio={err / max(floor, 1e-30):.2f} vs_rounded={err_r:.3e}"


def check_fwd(w, inp, o_gpu, lse_gpu, rows=None):
    """Full-tensor forward parity; returns list of (ok, msg)."""
    rin = workloads.rounded(inp, w.dtype)
    kw = oracle_kwargs(w, inp)
    o_m, l_m = oracle.fwd(inp["q"], inp["k"], inp["v"], **kw)
    o_r, l_r = oracle.fwd(rin["q"], rin["k"], rin["v"], **kw)
    res = [judge("O", o_gpu, o_m, o_r, w.dtype, O_CAP[w.dtype]),
           judge("LSE", lse_gpu, l_m, l_r, w.dtype, LSE_CAP, round_out=False)]
    empty = np.isneginf(l_r)
    if empty.any():
        res.append((bool(np.all(np.isneginf(lse_gpu[empty]))), "empty rows have LSE = -inf"))
    return res


def check_bwd(w, inp, dq, dk, dv):
    """Full-tensor backward parity on the gradients; returns list of (ok, msg)."""
    rin = workloads.rounded(inp, w.dtype)
    kw = oracle_kwargs(w, inp)
    m = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], **kw)
    r = oracle.bwd(rin["q"], rin["k"], rin["v"], rin["do"], **kw)
    return [
        judge("dQ", dq, m["dq"], r["dq"], w.dtype),
        judge("dK", dk, m["dk"], r["dk"], w.dtype),
        judge("dV", dv, m["dv"], r["dv"], w.dtype),
    ]
