"""Parity helpers: run the CUDA path and the float64 oracle on the same seeded
inputs and apply the acceptance rule.

Rule (TransformerEngine PR #3527, "Verification": the criterion FlashAttention
applies to itself, err(kernel, fp64) <= 2 * err(inputs rounded to dtype, fp64),
with the floor measured per case), read as:
  R      = oracle on the float64 master inputs
  floor  = max |round_to_dtype(oracle on dtype-rounded inputs) - R|  per tensor
           (the best a kernel with dtype inputs and dtype outputs could do;
           LSE is float32, so it is not rounded)
  pass   iff max |kernel - R| <= 2 * floor over every item (one row of one
           head) of the tensor that is not an edge item.
Edge items, found from the oracle's own mask (an oracle run with zero scores
gives LSE = ln(number of allowed keys)):
  * query rows (O, LSE, dQ) that see one to three keys, where the kernel's
    16-bit rounding of P and dS for the MMAs (absent from the floor)
    dominates; and key rows (dK, dV) that such a query row attends;
  * every item of a tensor whose floor is exactly 0 (e.g. dQ when every row
    sees one key), which no finite-precision kernel can meet.
  Edge items pass iff their error is <= 2 * floor + u * max|R|, u the unit
  roundoff of the output format (2^-8 bf16, 2^-11 fp16, 2^-24 for the fp32
  LSE), and never below 1e-5.
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
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nanmax(d)) if d.size else 0.0


UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11, "fp32": 2.0 ** -24}


def _item_err(got, ref):
    """|got - ref| elementwise (0 where both are the same infinity)."""
    a, b = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return d


def check_tensor(name, got, ref_master, ref_rounded, dtype, cap=None, round_out=True, edge=None):
    """Returns (ok, message) for one tensor.

    `edge` marks the edge items (boolean, the tensor's shape without its last
    axis, or the tensor's own shape for the per-row LSE); None = no edge
    items. Items that are not edge items must meet err <= 2 * floor; edge
    items get the margin u * max|R| (at least 1e-5), as does every item when
    the tensor's floor is exactly 0."""
    got = np.asarray(got, dtype=np.float64)
    ref_master = np.asarray(ref_master, dtype=np.float64)
    floor_src = workloads.round_to(ref_rounded, dtype) if round_out else ref_rounded
    floor = max_abs(floor_src, ref_master)
    d = _item_err(got, ref_master)
    per_item = d if d.ndim == 0 or edge is None or np.shape(edge) == d.shape else np.nanmax(d, axis=-1)
    if edge is None:
        edge_m = np.zeros(np.shape(per_item), dtype=bool)
    else:
        edge_m = np.broadcast_to(np.asarray(edge, dtype=bool), np.shape(per_item))
    if floor == 0.0:
        edge_m = np.ones(np.shape(per_item), dtype=bool)
    err = float(np.nanmax(per_item)) if per_item.size else 0.0
    strict = per_item[~edge_m]
    loose = per_item[edge_m]
    err_s = float(np.nanmax(strict)) if strict.size else 0.0
    err_e = float(np.nanmax(loose)) if loose.size else 0.0
    err_r = max_abs(got, ref_rounded)
    finite = np.isfinite(ref_master)
    rmax = float(np.max(np.abs(ref_master[finite]))) if np.any(finite) else 0.0
    u = UNIT_ROUNDOFF[dtype if round_out else "fp32"]
    bound_s = 2.0 * floor
    bound_e = max(2.0 * floor + u * rmax, 1e-5)
    ok = err_s <= bound_s and err_e <= bound_e and bool(np.all(np.isfinite(got) | np.isinf(ref_rounded)))
    if cap is not None:
        ok = ok and err_r <= cap
    msg = (f"{name}: err={err:.3e} floor={floor:.3e} ratio={err_s / max(floor, 1e-30):.2f} "
           f"({strict.size} items, bound 2*floor={bound_s:.3e})")
    if loose.size:
        msg += f" edge: {loose.size} items err={err_e:.3e} ratio={err_e / max(floor, 1e-30):.2f} bound={bound_e:.3e}"
    msg += f" vs_rounded={err_r:.3e}"
    return ok, msg


def _zeros_d1(x):
    return np.zeros(np.shape(x)[:-1] + (1,))


def allowed_keys(w, inp):
    """Keys each query row may attend, token-major [rows_q, Hq], from the
    oracle's mask: with all scores zero its LSE is ln(number of allowed keys)
    (one-wide rows keep it cheap)."""
    kw = oracle_kwargs(w, inp)
    _, lse = oracle.fwd(_zeros_d1(inp["q"]), _zeros_d1(inp["k"]), _zeros_d1(inp["k"]), **kw)
    return np.rint(np.exp(lse)).astype(np.int64)


EDGE_KEYS = 4  # query rows that see fewer allowed keys are edge items


def edge_items(w, inp, backward=True):
    """(query-side edge items [rows_q, Hq], key-side edge items [rows_kv, Hkv]
    or None): query rows with one to three allowed keys, and the keys such a
    row attends (an oracle backward with zero scores and dO marking the edge
    rows gives dV_j > 0 exactly for those keys)."""
    n = allowed_keys(w, inp)
    q_edge = n < EDGE_KEYS
    if not backward:
        return q_edge, None
    kw = oracle_kwargs(w, inp)
    mark = (q_edge & (n > 0)).astype(np.float64).reshape(np.shape(inp["q"])[:-2] + (w.heads_q, 1))
    z = _zeros_d1(inp["k"])
    r = oracle.bwd(_zeros_d1(inp["q"]), z, z, mark, **kw)
    k_edge = r["dv"][..., 0] > 0
    return q_edge, k_edge.reshape(-1, w.heads_kv)


def _q_items(edge_q, x, heads):
    """Edge items of a query-side tensor x (O or dQ) in its own layout."""
    return None if edge_q is None else edge_q.reshape(np.shape(x)[:-2] + (heads,))


def report(case, results):
    """Print every tensor's ratio line for `case`, then assert all passed."""
    for ok, msg in results:
        print(f"[{case}] {'ok  ' if ok else 'FAIL'} {msg}")
    assert all(ok for ok, _ in results), [m for ok, m in results if not ok]


def check_fwd(w, inp, o_gpu, lse_gpu, rows=None):
    """Full-tensor forward parity; returns list of (ok, msg)."""
    rin = workloads.rounded(inp, w.dtype)
    kw = oracle_kwargs(w, inp)
    o_m, l_m = oracle.fwd(inp["q"], inp["k"], inp["v"], **kw)
    o_r, l_r = oracle.fwd(rin["q"], rin["k"], rin["v"], **kw)
    eq, _ = edge_items(w, inp, backward=False)
    res = [check_tensor("O", o_gpu, o_m, o_r, w.dtype, O_CAP[w.dtype], edge=_q_items(eq, o_m, w.heads_q)),
           check_tensor("LSE", lse_gpu, l_m, l_r, w.dtype, LSE_CAP, round_out=False, edge=eq)]
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
    eq, ek = edge_items(w, inp)
    ekk = ek.reshape(np.shape(m["dk"])[:-2] + (w.heads_kv,))
    return [
        check_tensor("dQ", dq, m["dq"], r["dq"], w.dtype, edge=_q_items(eq, m["dq"], w.heads_q)),
        check_tensor("dK", dk, m["dk"], r["dk"], w.dtype, edge=ekk),
        check_tensor("dV", dv, m["dv"], r["dv"], w.dtype, edge=ekk),
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
    """(b, g, j) key rows of two kv heads of one sequence: the longest THD
    sequence (so long-sequence key tiles are checked), else the last batch
    entry; sequence edges, 128-row tile edges and random keys."""
    rng = np.random.Generator(np.random.PCG64(seed))
    _, lk = seq_lens(w, inp)
    b = int(np.argmax(lk)) if w.layout == "thd" else len(lk) - 1
    heads = rng.permutation(w.heads_kv)[:2]
    L = int(lk[b])
    out = []
    for g in heads:
        keys = {0, L - 1, min(127, L - 1), min(128, L - 1), L // 2, max(L - 129, 0)}
        while len(keys) < min(n, L):
            keys.add(int(rng.integers(L)))
        out += [(b, int(g), j) for j in sorted(keys)]
    return np.array(out, dtype=np.int32)


def _sampled_edges(w, inp, bhi, bgj):
    """Edge items of sampled query rows (bhi) and key rows (bgj), from the
    oracle's mask with one-wide zero rows (see edge_items)."""
    kw = oracle_kwargs(w, inp)
    zq, zk = _zeros_d1(inp["q"]), _zeros_d1(inp["k"])
    _, lse = oracle.fwd_rows(zq, zk, zk, bhi, **kw)
    q_edge = np.rint(np.exp(lse)) < EDGE_KEYS
    if bgj is None:
        return q_edge, None
    k_edge = np.zeros(len(bgj), dtype=bool)
    kt = np.array([kv_token_row(w, inp, b, j) for b, _, j in bgj])
    for b, g in sorted({(int(b), int(g)) for b, g, _ in bgj}):
        part = dict(batch_range=(b, b + 1), kv_head_range=(g, g + 1))
        r0 = oracle.bwd(zq, zk, zk, np.zeros(np.shape(zq)), **kw, **part)
        n = np.rint(np.exp(r0["lse"]))  # -inf (rows outside the part) -> 0
        mark = ((n > 0) & (n < EDGE_KEYS)).astype(np.float64).reshape(np.shape(zq))
        r1 = oracle.bwd(zq, zk, zk, mark, **kw, **part)
        dv = r1["dv"].reshape(-1, w.heads_kv)
        sel = (bgj[:, 0] == b) & (bgj[:, 1] == g)
        k_edge[sel] = dv[kt[sel], g] > 0
    return q_edge, k_edge


def check_sampled(w, inp, out, n_rows=40, n_keys=12, seed=0, backward=True):
    """Parity on sampled rows of a full-size run. `out` holds the GPU results
    as float64 numpy arrays in their layouts: o, lse and (backward) dq, dk, dv."""
    rin = workloads.rounded(inp, w.dtype)
    kw = oracle_kwargs(w, inp)
    bhi = sample_rows(w, inp, n_rows, seed)
    bgj = sample_keys(w, inp, n_keys, seed) if backward else None
    q_edge, k_edge = _sampled_edges(w, inp, bhi, bgj)
    tr = [token_row(w, inp, b, i) for b, _, i in bhi]
    o_m, l_m = oracle.fwd_rows(inp["q"], inp["k"], inp["v"], bhi, **kw)
    o_r, l_r = oracle.fwd_rows(rin["q"], rin["k"], rin["v"], bhi, **kw)
    nh = w.heads_q
    o_g = np.stack([out["o"].reshape(-1, nh, w.dv)[t, h] for t, (_, h, _) in zip(tr, bhi)])
    l_g = np.array([out["lse"][t, h] for t, (_, h, _) in zip(tr, bhi)])
    res = [check_tensor("O", o_g, o_m, o_r, w.dtype, O_CAP[w.dtype], edge=q_edge),
           check_tensor("LSE", l_g, l_m, l_r, w.dtype, LSE_CAP, round_out=False, edge=q_edge)]
    if not backward:
        return res
    dq_m = oracle.dq_rows(inp["q"], inp["k"], inp["v"], inp["do"], bhi, **kw)
    dq_r = oracle.dq_rows(rin["q"], rin["k"], rin["v"], rin["do"], bhi, **kw)
    dq_g = np.stack([out["dq"].reshape(-1, nh, w.head_dim)[t, h] for t, (_, h, _) in zip(tr, bhi)])
    res.append(check_tensor("dQ", dq_g, dq_m, dq_r, w.dtype, edge=q_edge))
    kt = [kv_token_row(w, inp, b, j) for b, _, j in bgj]
    dk_m, dv_m = oracle.dkdv_rows(inp["q"], inp["k"], inp["v"], inp["do"], bgj, **kw)
    dk_r, dv_r = oracle.dkdv_rows(rin["q"], rin["k"], rin["v"], rin["do"], bgj, **kw)
    nkv = w.heads_kv
    dk_g = np.stack([out["dk"].reshape(-1, nkv, w.head_dim)[t, g] for t, (_, g, _) in zip(kt, bgj)])
    dv_g = np.stack([out["dv"].reshape(-1, nkv, w.head_dim)[t, g] for t, (_, g, _) in zip(kt, bgj)])
    res.append(check_tensor("dK", dk_g, dk_m, dk_r, w.dtype, edge=k_edge))
    res.append(check_tensor("dV", dv_g, dv_m, dv_r, w.dtype, edge=k_edge))
    return res
