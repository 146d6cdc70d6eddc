"""Forward parity: the CUDA path through the C ABI vs the float64 oracle.

Sizes are small enough for the oracle to finish in seconds while spanning
several 128-row tiles and a ragged tail; the cases cover every layout, mask,
GQA, windows, head_dim 128/256/512 and rows with no allowed key.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

FWD_CASES = [
    workloads.TINY,
    Workload("bshd_gqa_ragged", "bshd", "causal", 2, 300, 300, 4, 2, 128, "bf16"),
    Workload("sbhd_fp16_nomask", "sbhd", "none", 2, 200, 200, 2, 2, 128, "fp16", std=0.5),
    Workload("thd_varlen", "thd", "causal", 4, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300)),
    Workload("bottom_right_rect", "bshd", "causal_br", 1, 200, 333, 2, 1, 128, "bf16"),
    Workload("window_d256", "bshd", "causal", 1, 400, 400, 2, 1, 256, "bf16", window=(100, 0)),
    Workload("d512_br", "bshd", "causal_br", 1, 130, 300, 2, 1, 512, "bf16"),
    Workload("d512_nomask", "bshd", "none", 1, 129, 257, 2, 2, 512, "bf16"),
    Workload("br_more_queries_than_keys", "bshd", "causal_br", 1, 300, 140, 2, 2, 128, "bf16"),
    Workload("d256_fp16_sbhd_window", "sbhd", "causal", 2, 260, 260, 2, 1, 256, "fp16", window=(64, 0)),
    Workload("d512_fp16_br", "bshd", "causal_br", 1, 200, 333, 2, 1, 512, "fp16", std=0.5),
    Workload("d512_thd_varlen", "thd", "causal", 3, 260, 260, 2, 1, 512, "bf16", len_range=(1, 260)),
    # windows at every head dim: two-sided (no causal mask, Sq == Sk), causal at D512, and a
    # left window measured from the bottom-right diagonal
    Workload("d256_two_sided_window", "bshd", "none", 1, 300, 300, 2, 2, 256, "bf16", window=(70, 45)),
    Workload("d512_causal_window", "bshd", "causal", 1, 400, 400, 2, 1, 512, "bf16", window=(150, 0)),
    Workload("d512_two_sided_window_gqa", "bshd", "none", 1, 260, 260, 4, 2, 512, "bf16", window=(40, 90)),
    Workload("br_window_d128", "bshd", "causal_br", 1, 200, 333, 2, 1, 128, "bf16", window=(60, 0)),
    Workload("br_window_d256", "bshd", "causal_br", 1, 200, 333, 2, 1, 256, "bf16", window=(90, 0)),
    # a diagonal-only window: every row sees its own key alone (P = 1, O = V)
    Workload("diagonal_window_d128", "bshd", "causal", 1, 300, 300, 2, 2, 128, "bf16", window=(0, 0)),
    Workload("diagonal_window_d256", "bshd", "causal", 1, 300, 300, 2, 1, 256, "bf16", window=(0, 0)),
    Workload("diagonal_window_d512", "bshd", "causal", 1, 300, 300, 2, 1, 512, "bf16", window=(0, 0)),
]


def run_fwd(w, inp):
    from scaled_dot_product_02_gb300 import sdpa_fwd, sdpa_get_device_error
    from parity import gpu_kwargs, to_device, report

    q, k, v = (to_device(inp[x], w.dtype) for x in ("q", "k", "v"))
    o, lse = sdpa_fwd(q, k, v, **gpu_kwargs(w, inp))
    assert sdpa_get_device_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("w", FWD_CASES, ids=lambda w: w.name)
def test_forward_matches_oracle(w):
    from parity import check_fwd, report

    inp = workloads.make_inputs(w, seed=7)
    o, lse = run_fwd(w, inp)
    results = check_fwd(w, inp, o, lse)
    report(w.name, results)
