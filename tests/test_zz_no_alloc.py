"""sdpa_bwd_noalloc: the backward for callers that cannot allocate device
memory (its scratch is the library's static device array). It must give the
same gradients as sdpa_bwd with a caller-provided workspace, call after call:
two calls in a row, on two different problems so that the second runs over
what the first left in the shared array, both pass the oracle parity rule and
match sdpa_bwd -- dK/dV bit for bit, and dQ bit for bit too where it is
deterministic (head_dim 256, or deterministic = 1), else (fp32 reductions)
to within one bf16 rounding. The cases cover every path that keeps scratch in
the array: the head_dim 128 accumulator, the deterministic head_dim 128
backward, and the head_dim 256 P/dS tile arrays (one and several key
chunks). This file sorts last so a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

# (first problem, second problem, deterministic, kv_chunk): the first is the
# larger one, so the second call finds the first call's data in the array
CASES = {
    "d128_thd_gqa": (Workload("noalloc_thd_gqa_a", "thd", "causal", 3, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300)),
                     Workload("noalloc_thd_gqa_b", "thd", "causal", 2, 200, 200, 4, 2, 128, "bf16", len_range=(1, 200)),
                     False, 0),
    "d128_deterministic": (Workload("noalloc_det_a", "bshd", "causal", 2, 300, 300, 4, 2, 128, "bf16"),
                           Workload("noalloc_det_b", "thd", "causal", 2, 250, 250, 4, 1, 128, "bf16", len_range=(1, 250)),
                           True, 0),
    "d256_bshd": (Workload("noalloc_d256_a", "bshd", "causal", 1, 384, 384, 2, 1, 256, "bf16"),
                  Workload("noalloc_d256_b", "bshd", "causal_br", 1, 200, 300, 2, 2, 256, "bf16"),
                  False, 0),
    "d256_key_chunks": (Workload("noalloc_d256_chunks_a", "bshd", "none", 1, 256, 512, 2, 1, 256, "bf16"),
                        Workload("noalloc_d256_chunks_b", "bshd", "causal", 1, 300, 300, 2, 1, 256, "bf16"),
                        False, 128),
}


def _one_call(w, seed, deterministic, kv_chunk):
    import torch

    import scaled_dot_product_02_gb300 as sdpa
    from parity import check_bwd, gpu_kwargs, report, to_device

    inp = workloads.make_inputs(w, seed=seed)
    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa.sdpa_fwd(q, k, v, **kw)
    ref = sdpa.sdpa_bwd(q, k, v, o, lse, do, deterministic=deterministic, kv_chunk=kv_chunk, **kw)
    torch.cuda.synchronize()
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
    sdpa.sdpa_bwd_noalloc(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, deterministic=deterministic, kv_chunk=kv_chunk,
                          **kw)
    assert sdpa.sdpa_get_device_error() == 0
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), f"{w.name}: dK/dV differ from sdpa_bwd"
    if deterministic or w.head_dim != 128:
        assert torch.equal(dq, ref[0]), f"{w.name}: dQ differs from sdpa_bwd"
    else:
        diff = (dq.float() - ref[0].float()).abs().max().item()
        assert diff <= 2.0 ** -8 * max(1.0, ref[0].float().abs().max().item()), f"{w.name}: dQ differs by {diff}"
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    report(f"{w.name} (no allocation)", check_bwd(w, inp, f(dq), f(dk), f(dv)))


def _workspace_bytes(w, seed, deterministic, kv_chunk):
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    lens = workloads.thd_lengths(w, seed) if w.layout == "thd" else None
    sq, sk = workloads.shapes(w, lens, lens)
    p = sdpa.make_problem(torch.empty(sq, dtype=torch.bfloat16), torch.empty(sk, dtype=torch.bfloat16),
                          layout=w.layout, mask=w.mask, batch=w.batch if w.layout == "thd" else None,
                          max_seqlen_q=w.seqlen_q, max_seqlen_kv=w.seqlen_kv, deterministic=deterministic,
                          kv_chunk=kv_chunk)
    return sdpa.sdpa_bwd_workspace_size(p)


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_backward_matches_workspace_backward_twice(case):
    import scaled_dot_product_02_gb300 as sdpa

    first, second, det, chunk = CASES[case]
    for w in (first, second):
        assert 0 < _workspace_bytes(w, 51, det, chunk) <= sdpa.NOALLOC_MAX_BYTES, w.name
    _one_call(first, 51, det, chunk)
    _one_call(second, 51, det, chunk)


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
