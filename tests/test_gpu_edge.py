"""Degenerate shapes and failure paths on the GPU.

* Parity on shapes at the edges of the tiling and masking logic: a single
  query or key, window 0 (diagonal only), two-sided windows, scales far from
  1/sqrt(D), a 16:1 GQA ratio, many tiny THD sequences and empty ones.
* The THD metadata guard (TransformerEngine PR #3705: compactness is checked
  on the GPU on every execution): corrupted cu_seqlens made on the host are
  reported as SDPA_ERR_BAD_SEQLENS and no output is written.
* The bounded waits: a wait on a barrier nothing arrives on reports
  SDPA_ERR_TIMEOUT and the context stays usable.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

EDGE = [
    Workload("one_query", "bshd", "none", 2, 1, 200, 2, 1, 128, "bf16"),
    Workload("one_key", "bshd", "causal_br", 1, 130, 1, 2, 2, 128, "bf16"),
    Workload("diagonal_only", "bshd", "causal", 1, 200, 200, 2, 2, 128, "bf16", window=(0, 0)),
    Workload("two_sided_window", "bshd", "none", 1, 300, 300, 2, 2, 128, "bf16", window=(20, 37)),
    Workload("gqa_16_to_1", "bshd", "causal", 1, 256, 256, 16, 1, 128, "bf16"),
    Workload("tiny_thd_sequences", "thd", "causal", 40, 3, 3, 2, 1, 128, "bf16", len_range=(1, 3)),
    Workload("fp16_nomask_d256", "bshd", "none", 1, 140, 140, 2, 2, 256, "fp16", std=0.5),
]


def _run(w, inp, scale=None):
    from parity import gpu_kwargs, to_device, report
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    if scale is not None:
        kw["scale"] = scale
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, **kw)
    assert sdpa_get_device_error() == 0
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f(o), lse.cpu().numpy().astype(np.float64), f(dq), f(dk), f(dv)


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_edge_shapes_match_oracle(w):
    from parity import check_bwd, check_fwd, report

    inp = workloads.make_inputs(w, seed=5)
    o, lse, dq, dk, dv = _run(w, inp)
    res = check_fwd(w, inp, o, lse) + check_bwd(w, inp, dq, dk, dv)
    report(w.name, res)


@pytest.mark.parametrize("scale", [0.02, 0.35])
def test_other_softmax_scales(scale):
    import parity

    w = Workload("scaled", "bshd", "causal", 1, 200, 200, 2, 2, 128, "bf16")
    inp = workloads.make_inputs(w, seed=6)
    o, lse, dq, dk, dv = _run(w, inp, scale=scale)
    ws = _ScaledWorkload(w, scale)
    res = parity.check_fwd(ws, inp, o, lse) + parity.check_bwd(ws, inp, dq, dk, dv)
    parity.report(w.name, res)


class _ScaledWorkload:
    """A workload view whose softmax scale is overridden (for the oracle)."""

    def __init__(self, w, scale):
        self._w, self.scale = w, scale

    def __getattr__(self, name):
        return getattr(self._w, name)


def test_empty_thd_sequences_are_allowed():
    from parity import check_bwd, check_fwd, report

    w = Workload("thd_with_empty", "thd", "causal", 4, 150, 150, 2, 2, 128, "bf16")
    inp = workloads.make_inputs(w, seed=8, lengths=np.array([150, 0, 37, 0]))
    o, lse, dq, dk, dv = _run(w, inp)
    res = check_fwd(w, inp, o, lse) + check_bwd(w, inp, dq, dk, dv)
    report(w.name, res)


BAD_CU = {
    "nonzero_start": ([1, 100, 200], [0, 100, 200]),
    "decreasing": ([0, 120, 100], [0, 100, 200]),
    "wrong_total": ([0, 100, 190], [0, 100, 190]),
    "live_q_empty_kv": ([0, 100, 200], [0, 100, 100]),
    "longer_than_declared": ([0, 10, 200], [0, 10, 200]),
}


@pytest.mark.parametrize("case", sorted(BAD_CU))
def test_guard_rejects_bad_cu_seqlens_and_writes_nothing(case):
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    cu_q, cu_kv = (torch.tensor(x, dtype=torch.int32, device="cuda") for x in BAD_CU[case])
    total = 200
    q = torch.randn(total, 2, 128, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(total, 2, 128, device="cuda", dtype=torch.bfloat16)
    v = torch.randn_like(k)
    o = torch.full_like(q, 7.0)
    lse = torch.full((total, 2), 7.0, device="cuda")
    kw = dict(layout="thd", mask="causal", cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, max_seqlen_q=100,
              max_seqlen_kv=100)
    sdpa.sdpa_fwd(q, k, v, out=o, lse=lse, **kw)
    assert sdpa.sdpa_get_device_error() == 6  # SDPA_ERR_BAD_SEQLENS
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)
    dq, dk, dv = (torch.full_like(x, 7.0) for x in (q, k, v))
    sdpa.sdpa_bwd(q, k, v, o, lse, q, dq=dq, dk=dk, dv=dv, **kw)
    assert sdpa.sdpa_get_device_error() == 6
    assert torch.all(dq == 7.0) and torch.all(dk == 7.0) and torch.all(dv == 7.0)
    # the next valid call runs normally
    good = torch.tensor([0, 100, 200], dtype=torch.int32, device="cuda")
    kw.update(cu_seqlens_q=good, cu_seqlens_kv=good)
    sdpa.sdpa_fwd(q, k, v, out=o, lse=lse, **kw)
    assert sdpa.sdpa_get_device_error() == 0
    assert torch.isfinite(o.float()).all()


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    assert sdpa.sdpa_get_device_error() == 0
    sdpa.sdpa_selftest_bounded_wait(20000)  # 20 ms on a barrier nothing arrives on
    assert sdpa.sdpa_get_device_error() == 7  # SDPA_ERR_TIMEOUT, then cleared
    assert sdpa.sdpa_get_device_error() == 0
    q = torch.randn(1, 128, 2, 128, device="cuda", dtype=torch.bfloat16)
    o, lse = sdpa.sdpa_fwd(q, q, q, mask="causal")
    assert sdpa.sdpa_get_device_error() == 0
    assert torch.isfinite(o.float()).all()
