"""The head_dim 256/512 backward with its keys split into chunks
(sdpa_problem.kv_chunk; TransformerEngine PR #3527, "Known limitations": a
workspace that grows with the key length caps the context, so the score
tiles are held one chunk of keys at a time).

Small chunks force several chunks on shapes the oracle checks in seconds:
  * parity against the float64 oracle under the per-case floor rule;
  * dK and dV are final after the chunk that holds their keys and are formed
    from the same tiles in the same order as with one chunk: bit for bit
    equal to the one-chunk backward;
  * dQ is summed over the chunks in a fixed order: two runs are bit for bit
    equal.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("d256_causal_5_chunks", "bshd", "causal", 1, 600, 600, 4, 2, 256, "bf16"), 128),
    (Workload("d256_window_chunks", "bshd", "causal", 1, 700, 700, 2, 1, 256, "bf16", window=(150, 0)), 256),
    (Workload("d256_fp16_sbhd_nomask", "sbhd", "none", 2, 300, 520, 2, 2, 256, "fp16", std=0.5), 384),
    (Workload("d512_br_rect_chunks", "bshd", "causal_br", 1, 200, 700, 2, 1, 512, "bf16"), 256),
    (Workload("d512_nomask_gqa_chunks", "bshd", "none", 1, 260, 390, 4, 2, 512, "bf16"), 128),
    (Workload("d512_thd_varlen_chunks", "thd", "causal", 3, 400, 400, 2, 1, 512, "bf16", len_range=(1, 400)), 128),
]


def _run(w, inp, kv_chunk):
    from parity import gpu_kwargs, to_device
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    grads = sdpa_bwd(q, k, v, o, lse, do, kv_chunk=kv_chunk, **kw)
    assert sdpa_get_device_error() == 0
    return grads


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_chunked_backward_matches_oracle_and_one_chunk(case):
    import torch

    from parity import check_bwd, report

    w, chunk = case
    inp = workloads.make_inputs(w, seed=41)
    dq, dk, dv = _run(w, inp, chunk)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    report(f"{w.name} kv_chunk={chunk}", check_bwd(w, inp, f(dq), f(dk), f(dv)))
    dq1, dk1, dv1 = _run(w, inp, 0)
    assert torch.equal(dk, dk1) and torch.equal(dv, dv1), "dK/dV differ from the one-chunk backward"
    dq2, dk2, dv2 = _run(w, inp, chunk)
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2), "two chunked runs differ"
