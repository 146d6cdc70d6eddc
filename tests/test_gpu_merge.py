"""GPU parity of sdpa_merge, the log-sum-exp merge of partial results over a
split of the keys (TransformerEngine PR #3527 context parallelism, PR #3693
"neutral statistics for empty ragged ring blocks").

* The merge kernel against the float64 oracle merge on the same inputs
  (16-bit partial outputs, fp32 LSE), element by element: the kernel adds
  fp32 arithmetic and one output rounding, so |O - O_ref| <= u |O_ref| +
  1e-6 (u = 2^-8 bf16, 2^-11 fp16) and |LSE - LSE_ref| <= 2e-6 (1 + |LSE|).
* The whole split path: sdpa_fwd over each key block, then sdpa_merge,
  against the oracle's attention over all keys, under the pages' rule with
  the floor of this two-stage path (partials rounded to the dtype, merged,
  rounded again): err <= 2 * floor + u * max|R|, plus the absolute caps.
* Empty blocks are neutral whatever their rows hold, and an item whose
  blocks are all empty gets O = 0, LSE = -inf.
"""
import numpy as np
import pytest

import workloads
from oracle import oracle

pytestmark = pytest.mark.gpu

U = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _to(x, dtype):
    import torch

    return workloads.to_torch(x, dtype).cuda().contiguous()


@pytest.mark.parametrize("dtype,d,n_parts", [("bf16", 128, 2), ("bf16", 256, 3), ("fp16", 512, 4),
                                             ("bf16", 128, 1), ("fp16", 128, 7)])
def test_merge_kernel_matches_oracle_merge(dtype, d, n_parts):
    import torch

    from scaled_dot_product_02_gb300 import sdpa_get_device_error, sdpa_merge

    r = _rng(100 + d + n_parts)
    rows, heads = 333, 3
    po = workloads.round_to(r.standard_normal((n_parts, rows, heads, d)), dtype)
    pl = (r.standard_normal((n_parts, rows, heads)) * 4.0 + 30.0).astype(np.float32).astype(np.float64)
    if n_parts > 1:
        pl[1, ::5] = -np.inf       # blocks that saw no keys for some rows
    pl[:, 7] = -np.inf             # a row whose blocks are all empty
    o, lse = sdpa_merge(_to(po, dtype), torch.from_numpy(pl.astype(np.float32)).cuda())
    assert sdpa_get_device_error() == 0
    o_ref, l_ref = oracle.merge(po, pl)
    got = o.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.all(got[7] == 0.0) and np.all(np.isneginf(gl[7]))
    fin = np.isfinite(l_ref)
    assert np.all(np.abs(got - o_ref) <= U[dtype] * np.abs(o_ref) + 1e-6)
    assert np.all(np.abs(gl[fin] - l_ref[fin]) <= 2e-6 * (1.0 + np.abs(l_ref[fin])))


def test_empty_blocks_are_neutral_whatever_they_hold():
    import torch

    from scaled_dot_product_02_gb300 import sdpa_merge

    r = _rng(7)
    po = workloads.round_to(r.standard_normal((3, 64, 2, 128)), "bf16")
    pl = r.standard_normal((3, 64, 2)).astype(np.float32).astype(np.float64)
    pl[1] = -np.inf
    po_t = _to(po, "bf16")
    po_t[1] = float("inf")  # never read: the block is empty
    o, lse = sdpa_merge(po_t, torch.from_numpy(pl.astype(np.float32)).cuda())
    o2, lse2 = sdpa_merge(_to(po[[0, 2]], "bf16"), torch.from_numpy(pl[[0, 2]].astype(np.float32)).cuda())
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 256), ("bf16", 512)])
def test_forward_over_key_blocks_then_merge_equals_attention_over_all_keys(dtype, d):
    import torch

    from scaled_dot_product_02_gb300 import sdpa_fwd, sdpa_get_device_error, sdpa_merge

    w = workloads.Workload("split", "bshd", "none", 2, 200, 700, 4, 2, d, dtype)
    inp = workloads.make_inputs(w, seed=21)
    bounds = [(0, 128), (128, 450), (450, 700)]  # unequal blocks, one not a tile multiple
    q = _to(inp["q"], dtype)
    parts_o, parts_l = [], []
    for a, b in bounds:
        k = _to(inp["k"][:, a:b], dtype)
        v = _to(inp["v"][:, a:b], dtype)
        o, lse = sdpa_fwd(q, k, v, layout="bshd", mask="none", scale=w.scale)
        parts_o.append(o)
        parts_l.append(lse)
    o, lse = sdpa_merge(torch.stack(parts_o), torch.stack(parts_l))
    assert sdpa_get_device_error() == 0
    got = o.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)

    # R: float64 attention over all keys on the master inputs
    o_m, l_m = oracle.fwd(inp["q"], inp["k"], inp["v"], layout="bshd", mask="none", scale=w.scale)
    # floor of the two-stage path: oracle partials on dtype-rounded inputs,
    # rounded to the dtype, merged in float64, rounded again
    rin = workloads.rounded(inp, dtype)
    po, pl = [], []
    for a, b in bounds:
        ob, lb = oracle.fwd(rin["q"], rin["k"][:, a:b], rin["v"][:, a:b], layout="bshd", mask="none", scale=w.scale)
        po.append(workloads.round_to(ob, dtype))
        pl.append(lb.reshape(2, 200, 4))
    o_f, l_f = oracle.merge(np.stack(po), np.stack(pl))
    floor_o = np.max(np.abs(workloads.round_to(o_f, dtype) - o_m))
    floor_l = np.max(np.abs(l_f.reshape(-1, 4) - l_m))
    err_o = np.max(np.abs(got - o_m))
    err_l = np.max(np.abs(gl - l_m))
    bound_o = 2 * floor_o + U[dtype] * np.max(np.abs(o_m))
    bound_l = max(2 * floor_l + 2.0 ** -24 * np.max(np.abs(l_m)), 1e-5)
    assert err_o <= bound_o, (err_o, floor_o, bound_o)
    assert err_l <= bound_l, (err_l, floor_l, bound_l)
    # the absolute caps are against the reference on the dtype-rounded inputs (as in parity.check_fwd)
    assert np.max(np.abs(got - workloads.round_to(o_f, dtype))) <= {"bf16": 2e-2, "fp16": 4e-3}[dtype]
    assert np.max(np.abs(gl - l_f.reshape(-1, 4))) <= 1e-3
