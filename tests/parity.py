"""Parity helpers: run the CUDA path and the float64 oracle on the same seeded
inputs and apply the acceptance rule.

Rule (TransformerEngine PR #3527, "Verification": the criterion FlashAttention
applies to itself, err(kernel, fp64) <= 2 * err(inputs rounded to dtype, fp64),
with the floor measured per case), read as:
  R      = oracle on the float64 master inputs
  floor  = max |round_to_dtype(oracle on dtype-rounded inputs) - R|  per tensor
           (the best a kernel with dtype inputs and dtype outputs could do;
           LSE is float32, so it is not rounded)
  pass   iff max |kernel - R| <= 2 * floor + u * max|R|, per tensor, where u
           is the unit roundoff of the output format (2^-8 bf16, 2^-11 fp16,
           2^-24 for the float32 LSE), i.e. half an output ulp of the largest
           element, and never below 1e-5 (for exactly-zero references);
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


UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11, "fp32": 2.0 ** -24}


def judge(name, got, ref_master, ref_rounded, dtype, cap=None, round_out=True):
    """Returns (ok, message) for one tensor.

    bound = 2 * floor + u * max|R|, with u the unit roundoff of the output
    format (half an output ulp of the largest reference element), and at
    least 1e-5 for references that are exactly zero (e.g. dQ when every row
    sees one key), where the floor is 0 and no finite-precision kernel can
    meet the bare 2x rule."""
    floor_src = workloads.round_to(ref_rounded, dtype) if round_out else ref_rounded
    floor = max_abs(floor_src, ref_master)
    err = max_abs(got, ref_master)
    err_r = max_abs(got, ref_rounded)
    finite = np.isfinite(ref_master)
    rmax = float(np.max(np.abs(ref_master[finite]))) if np.any(finite) else 0.0
    u = UNIT_ROUNDOFF[dtype if round_out else "fp32"]
    bound = max(2.0 * floor + u * rmax, 1e-5)
    ok = err <= bound and bool(np.all(np.isfinite(got) | np.isinf(ref_rounded)))
    if cap is not None:
        ok = ok and err_r <= cap
    return ok, (f"{name}: err={err:.3e} floor={floor:.3e} ratio={err / max(floor, 1e-30):.2f} "
                f"bound={bound:.3e} vs_rounded={err_r:.3e}")


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


def token_row(w, inp, b, i):
    if w.layout == "bshd":
        return b * w.seqlen_q + i
    if w.layout == "sbhd":
        return i * w.batch + b
    return int(inp["cu_seqlens_q"][b]) + i


def kv_token_row(w, inp, b, j):
    if w.layout == "bshd":
        return b * w.seqlen_kv + j
    if w.layout == "sbhd":
        return j * w.batch + b
    return int(inp["cu_seqlens_kv"][b]) + j


def seq_lens(w, inp):
    if w.layout == "thd":
        return np.diff(inp["cu_seqlens_q"]), np.diff(inp["cu_seqlens_kv"])
    return np.full(w.batch, w.seqlen_q), np.full(w.batch, w.seqlen_kv)


def sample_rows(w, inp, n, seed):
    """(b, h, i) query rows: sequence starts and ends, 128-row tile edges, random."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lq, _ = seq_lens(w, inp)
    rows = set()
    for b in range(len(lq)):
        L = int(lq[b])
        if L == 0:
            continue
        for i in (0, L - 1, min(127, L - 1), min(128, L - 1), L // 2):
            rows.add((b, int(rng.integers(w.heads_q)), i))
    while len(rows) < n:
        b = int(rng.integers(len(lq)))
        if lq[b]:
            rows.add((b, int(rng.integers(w.heads_q)), int(rng.integers(lq[b]))))
    return np.array(sorted(rows), dtype=np.int32)


def sample_keys(w, inp, n, seed):
    """(b, g, j) key rows of one (sequence, kv head): the shortest sequence for
    THD, so the oracle's per-group pass stays cheap."""
    rng = np.random.Generator(np.random.PCG64(seed))
    _, lk = seq_lens(w, inp)
    b = int(np.argmin(lk)) if w.layout == "thd" else 0
    g = int(rng.integers(w.heads_kv))
    L = int(lk[b])
    keys = {0, L - 1, min(127, L - 1), min(128, L - 1), L // 2}
    while len(keys) < min(n, L):
        keys.add(int(rng.integers(L)))
    return np.array([(b, g, j) for j in sorted(keys)], dtype=np.int32)


def check_sampled(w, inp, out, n_rows=40, n_keys=12, seed=0, backward=True):
    """Parity on sampled rows of a full-size run. `out` holds the GPU results
    as float64 numpy arrays in their layouts: o, lse and (backward) dq, dk, dv."""
    rin = workloads.rounded(inp, w.dtype)
    kw = oracle_kwargs(w, inp)
    bhi = sample_rows(w, inp, n_rows, seed)
    tr = [token_row(w, inp, b, i) for b, _, i in bhi]
    o_m, l_m = oracle.fwd_rows(inp["q"], inp["k"], inp["v"], bhi, **kw)
    o_r, l_r = oracle.fwd_rows(rin["q"], rin["k"], rin["v"], bhi, **kw)
    nh = w.heads_q
    o_g = np.stack([out["o"].reshape(-1, nh, w.dv)[t, h] for t, (_, h, _) in zip(tr, bhi)])
    l_g = np.array([out["lse"][t, h] for t, (_, h, _) in zip(tr, bhi)])
    res = [judge("O", o_g, o_m, o_r, w.dtype, O_CAP[w.dtype]),
           judge("LSE", l_g, l_m, l_r, w.dtype, LSE_CAP, round_out=False)]
    if not backward:
        return res
    dq_m = oracle.dq_rows(inp["q"], inp["k"], inp["v"], inp["do"], bhi, **kw)
    dq_r = oracle.dq_rows(rin["q"], rin["k"], rin["v"], rin["do"], bhi, **kw)
    dq_g = np.stack([out["dq"].reshape(-1, nh, w.head_dim)[t, h] for t, (_, h, _) in zip(tr, bhi)])
    res.append(judge("dQ", dq_g, dq_m, dq_r, w.dtype))
    bgj = sample_keys(w, inp, n_keys, seed)
    kt = [kv_token_row(w, inp, b, j) for b, _, j in bgj]
    dk_m, dv_m = oracle.dkdv_rows(inp["q"], inp["k"], inp["v"], inp["do"], bgj, **kw)
    dk_r, dv_r = oracle.dkdv_rows(rin["q"], rin["k"], rin["v"], rin["do"], bgj, **kw)
    nkv = w.heads_kv
    dk_g = np.stack([out["dk"].reshape(-1, nkv, w.head_dim)[t, g] for t, (_, g, _) in zip(kt, bgj)])
    dv_g = np.stack([out["dv"].reshape(-1, nkv, w.head_dim)[t, g] for t, (_, g, _) in zip(kt, bgj)])
    res.append(judge("dK", dk_g, dk_m, dk_r, w.dtype))
    res.append(judge("dV", dv_g, dv_m, dv_r, w.dtype))
    return res
