"""Backward parity: dQ/dK/dV from the CUDA path (fed with its own forward's O
and LSE) against the float64 oracle, under the same per-case floor rule."""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

BWD_CASES = [
    workloads.TINY,
    Workload("bshd_gqa_ragged", "bshd", "causal", 2, 300, 300, 4, 2, 128, "bf16"),
    Workload("sbhd_fp16_nomask", "sbhd", "none", 2, 200, 200, 2, 2, 128, "fp16", std=0.5),
    Workload("thd_varlen_gqa", "thd", "causal", 4, 300, 300, 4, 1, 128, "bf16", len_range=(1, 300)),
    Workload("bottom_right_rect", "bshd", "causal_br", 1, 200, 333, 2, 1, 128, "bf16"),
    Workload("window_d128", "bshd", "causal", 1, 400, 400, 2, 2, 128, "bf16", window=(100, 0)),
    Workload("br_more_queries_than_keys", "bshd", "causal_br", 1, 300, 140, 2, 2, 128, "bf16"),
    # head_dim 256 / 512: two-phase backward (score tiles + GEMMs)
    Workload("window_d256", "bshd", "causal", 1, 400, 400, 2, 1, 256, "bf16", window=(100, 0)),
    Workload("d256_fp16_sbhd_window", "sbhd", "causal", 2, 260, 260, 2, 1, 256, "fp16", window=(64, 0)),
    Workload("window_d256_gqa_three_kv_heads", "bshd", "causal", 1, 450, 450, 6, 3, 256, "bf16", window=(150, 0)),
    Workload("d256_thd_varlen", "thd", "causal", 3, 300, 300, 4, 2, 256, "bf16", len_range=(1, 300)),
    Workload("d512_br", "bshd", "causal_br", 1, 130, 300, 2, 1, 512, "bf16"),
    Workload("d512_nomask_gqa", "bshd", "none", 1, 129, 257, 4, 2, 512, "bf16"),
    Workload("d512_br_more_queries", "bshd", "causal_br", 1, 300, 140, 2, 2, 512, "bf16"),
    Workload("d512_fp16_br", "bshd", "causal_br", 1, 200, 333, 2, 1, 512, "fp16", std=0.5),
    Workload("d512_thd_varlen", "thd", "causal", 3, 260, 260, 2, 1, 512, "bf16", len_range=(1, 260)),
    Workload("d256_fp16_thd_nomask", "thd", "none", 3, 200, 200, 2, 2, 256, "fp16", len_range=(1, 200)),
    # windows at every head dim: two-sided (no causal mask, Sq == Sk), causal at D512, and a
    # left window measured from the bottom-right diagonal
    Workload("d256_two_sided_window", "bshd", "none", 1, 300, 300, 2, 2, 256, "bf16", window=(70, 45)),
    Workload("d512_causal_window", "bshd", "causal", 1, 400, 400, 2, 1, 512, "bf16", window=(150, 0)),
    Workload("d512_two_sided_window_gqa", "bshd", "none", 1, 260, 260, 4, 2, 512, "bf16", window=(40, 90)),
    Workload("br_window_d128", "bshd", "causal_br", 1, 200, 333, 2, 1, 128, "bf16", window=(60, 0)),
    Workload("br_window_d256", "bshd", "causal_br", 1, 200, 333, 2, 1, 256, "bf16", window=(90, 0)),
    # a diagonal-only window: every row sees its own key alone (P = 1, so dS, dQ and dK vanish and
    # dV = dO). The kernels' dQ and dK are then the rounding residues of dP - delta (two fp32 sums of
    # the same D products), held to the 1e-5 margin of a tensor whose reference is exactly zero;
    # std 0.5 keeps those products, and so the residues, at a quarter of unit-variance inputs' at
    # head_dim 256 and 512
    Workload("diagonal_window_d128", "bshd", "causal", 1, 300, 300, 2, 2, 128, "bf16", window=(0, 0)),
    Workload("diagonal_window_d256", "bshd", "causal", 1, 300, 300, 2, 1, 256, "bf16", window=(0, 0), std=0.5),
    Workload("diagonal_window_d512", "bshd", "causal", 1, 300, 300, 2, 1, 512, "bf16", window=(0, 0), std=0.5),
]


def run_fwd_bwd(w, inp):
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error
    from parity import gpu_kwargs, to_device, report

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, **kw)
    assert sdpa_get_device_error() == 0
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f(dq), f(dk), f(dv)


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: w.name)
def test_backward_matches_oracle(w):
    from parity import check_bwd, report

    inp = workloads.make_inputs(w, seed=11)
    dq, dk, dv = run_fwd_bwd(w, inp)
    results = check_bwd(w, inp, dq, dk, dv)
    report(w.name, results)
