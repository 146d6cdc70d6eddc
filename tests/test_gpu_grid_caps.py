"""Race-detection stand-in: every attention kernel rerun with its CTAs capped
at 1, 2 and the SM count (sdpa_debug_set_max_ctas) must give the same bits.

TransformerEngine PR #3705 ("sync qualification") records a barrier-phase bug
in the dQ credit protocol that passed the numerical tests and only the race
checker caught. compute-sanitizer's race and sync checks are closed on this
pool, so the schedule is varied instead: with one CTA the persistent head_dim
128 forward walks every query tile through both of its pipelines, the
ticket queue and every barrier phase in one CTA; with one or two CTAs in
flight the other kernels run each work item with nothing beside it. O, LSE,
dK, dV (and dQ where it is deterministic: deterministic = 1, head_dim 256 and
512, the FP8 forward's O) are compared bit for bit with the uncapped run; dQ
of the default head_dim 128 backward, summed with fp32 reductions in
whatever order the CTAs reach them, to within one bf16 rounding.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("d128_thd_gqa", "thd", "causal", 4, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300)), False, 0),
    (Workload("d128_bshd_deterministic", "bshd", "causal_br", 1, 200, 333, 4, 1, 128, "bf16"), True, 0),
    (Workload("d256_window", "bshd", "causal", 1, 400, 400, 2, 1, 256, "bf16", window=(100, 0)), False, 0),
    (Workload("d512_br_chunks", "bshd", "causal_br", 1, 200, 520, 2, 1, 512, "bf16"), False, 128),
]


def _sm_count():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


def _run(w, inp, det, chunk):
    from parity import gpu_kwargs, to_device
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, deterministic=det, kv_chunk=chunk, **kw)
    assert sdpa_get_device_error() == 0
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_results_do_not_depend_on_how_many_ctas_run(case):
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    w, det, chunk = case
    inp = workloads.make_inputs(w, seed=71)
    ref = _run(w, inp, det, chunk)
    exact_dq = det or w.head_dim != 128
    try:
        for cap in (1, 2, _sm_count()):
            sdpa.sdpa_debug_set_max_ctas(cap)
            got = _run(w, inp, det, chunk)
            for name, a, b in zip(("O", "LSE", "dK", "dV"), (got[0], got[1], got[3], got[4]),
                                  (ref[0], ref[1], ref[3], ref[4])):
                assert torch.equal(a, b), f"{name} differs with at most {cap} CTAs"
            if exact_dq:
                assert torch.equal(got[2], ref[2]), f"dQ differs with at most {cap} CTAs"
            else:
                diff = (got[2].float() - ref[2].float()).abs().max().item()
                assert diff <= 2.0 ** -8 * max(1.0, ref[2].float().abs().max().item()), (cap, diff)
    finally:
        sdpa.sdpa_debug_set_max_ctas(0)


@pytest.mark.parametrize("head_dim", [128, 256])
@pytest.mark.parametrize("shape", ["thd_varlen", "diagonal_window"])
def test_fp8_forward_does_not_depend_on_how_many_ctas_run(head_dim, shape):
    """With one or two CTAs every CTA runs many tiles back to back; the
    diagonal window gives every query tile a single key tile, so at head_dim
    256 consecutive tiles reuse the row-stats slots as fast as they can."""
    import torch

    import scaled_dot_product_02_gb300 as sdpa
    from parity import gpu_kwargs

    if shape == "thd_varlen":
        w = Workload("fp8_thd", "thd", "causal", 3, 300, 300, 4, 2, head_dim, "bf16", len_range=(1, 300))
    else:
        w = Workload("fp8_diag", "bshd", "causal", 2, 600, 600, 4, 2, head_dim, "bf16", window=(0, 0))
    inp = workloads.fp8_inputs(w, seed=73)
    q8, k8, v8 = (torch.from_numpy(inp[x]).cuda() for x in ("q8", "k8", "v8"))
    kw = gpu_kwargs(w, inp)
    ref = sdpa.sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, **kw)
    try:
        for cap in (1, 2, _sm_count()):
            sdpa.sdpa_debug_set_max_ctas(cap)
            got = sdpa.sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, **kw)
            assert sdpa.sdpa_get_device_error() == 0
            assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), cap
    finally:
        sdpa.sdpa_debug_set_max_ctas(0)


def test_cap_is_validated():
    import scaled_dot_product_02_gb300 as sdpa

    with pytest.raises(sdpa.SdpaError):
        sdpa.sdpa_debug_set_max_ctas(-1)
    sdpa.sdpa_debug_set_max_ctas(0)
