"""The deterministic backward (sdpa_problem.deterministic = 1).

* Parity: dQ, dK, dV against the float64 oracle under the same per-case
  floor rule as the default backward, on the head_dim 128 cases (where a
  separate dQ pass replaces the fp32 reductions) and one head_dim 256 case
  (whose two-phase backward is deterministic either way).
* Reproducibility: two runs give bitwise identical dQ, dK and dV; the
  default head_dim 128 dQ agrees with it to within the parity rule, not
  bitwise.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

DET_CASES = [
    workloads.TINY,
    Workload("bshd_gqa_ragged", "bshd", "causal", 2, 300, 300, 4, 2, 128, "bf16"),
    Workload("sbhd_fp16_nomask", "sbhd", "none", 2, 200, 200, 2, 2, 128, "fp16", std=0.5),
    Workload("thd_varlen_gqa", "thd", "causal", 4, 300, 300, 4, 1, 128, "bf16", len_range=(1, 300)),
    Workload("bottom_right_rect", "bshd", "causal_br", 1, 200, 333, 2, 1, 128, "bf16"),
    Workload("window_d128", "bshd", "causal", 1, 400, 400, 2, 2, 128, "bf16", window=(100, 0)),
    Workload("br_more_queries_than_keys", "bshd", "causal_br", 1, 300, 140, 2, 2, 128, "bf16"),
    Workload("window_d256", "bshd", "causal", 1, 400, 400, 2, 1, 256, "bf16", window=(100, 0)),
]


def _run(w, inp, deterministic):
    from parity import gpu_kwargs, to_device
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    out = sdpa_bwd(q, k, v, o, lse, do, deterministic=deterministic, **kw)
    assert sdpa_get_device_error() == 0
    return out


@pytest.mark.parametrize("w", DET_CASES, ids=lambda w: w.name)
def test_deterministic_backward_matches_oracle(w):
    from parity import check_bwd

    inp = workloads.make_inputs(w, seed=11)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    dq, dk, dv = (f(t) for t in _run(w, inp, True))
    results = check_bwd(w, inp, dq, dk, dv)
    msgs = [m for _, m in results]
    print(w.name, msgs)
    assert all(ok for ok, _ in results), msgs


def test_two_deterministic_runs_are_bitwise_identical():
    import torch

    w = Workload("repro", "thd", "causal", 6, 700, 700, 8, 2, 128, "bf16", len_range=(200, 700))
    inp = workloads.make_inputs(w, seed=12)
    a = _run(w, inp, True)
    b = _run(w, inp, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    # the default path forms the same dQ up to the order of its fp32 reductions
    c = _run(w, inp, False)
    diff = (a[0].float() - c[0].float()).abs().max().item()
    assert diff <= 2.0 ** -7 * a[0].float().abs().max().item()
    assert torch.equal(a[1], c[1]) and torch.equal(a[2], c[2])  # dK, dV: the same kernel either way
