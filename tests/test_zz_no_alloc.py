"""sdpa_bwd_noalloc: the backward for callers that cannot allocate device
memory (its scratch is the library's static device array). It must give the
same gradients as sdpa_bwd with a caller-provided workspace, call after call:
two calls in a row both pass the oracle parity rule, their dK/dV equal
sdpa_bwd's bit for bit (those are deterministic), and dQ (accumulated with
fp32 atomics) agrees to within one bf16 rounding. This file sorts last so a
run that stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASE = Workload("noalloc_thd_gqa", "thd", "causal", 3, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300))


def test_noalloc_backward_matches_workspace_backward_twice():
    import torch

    import scaled_dot_product_02_gb300 as sdpa
    from parity import check_bwd, gpu_kwargs, to_device, report

    inp = workloads.make_inputs(CASE, seed=21)
    q, k, v, do = (to_device(inp[x], CASE.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(CASE, inp)
    o, lse = sdpa.sdpa_fwd(q, k, v, **kw)
    ref = sdpa.sdpa_bwd(q, k, v, o, lse, do, **kw)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    for call in range(2):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        sdpa.sdpa_bwd_noalloc(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, **kw)
        assert sdpa.sdpa_get_device_error() == 0
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), f"call {call}: dK/dV differ"
        diff = (dq.float() - ref[0].float()).abs().max().item()
        assert diff <= 2.0 ** -8 * max(1.0, ref[0].float().abs().max().item()), f"call {call}: dQ differs by {diff}"
        results = check_bwd(CASE, inp, f(dq), f(dk), f(dv))
        report(f"{CASE.name} call {call}", results)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    # 16 heads x 8192 rows x 128 x fp32 = 64 MiB of dQ accumulator > 32 MiB
    p = sdpa.make_problem(torch.empty(1, 8192, 16, 128, dtype=torch.bfloat16),
                          torch.empty(1, 128, 16, 128, dtype=torch.bfloat16), mask="causal")
    assert sdpa.sdpa_bwd_workspace_size(p) > sdpa.NOALLOC_MAX_BYTES
    null = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    rc = sdpa.lib().sdpa_bwd_noalloc(ctypes.byref(p), null, null, null, null, null, null, null, null, null, None,
                                     None, None)
    assert rc == 5  # SDPA_ERR_WORKSPACE_TOO_SMALL
