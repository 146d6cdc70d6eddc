"""CUDA-graph capture of the forward and backward.

sdpa_fwd and sdpa_bwd make no host synchronisation and no allocation (the
caller owns every buffer, the workspace included; TransformerEngine PR #3705,
"Execution and supported scope": the metadata guard runs on the GPU on every
execution, so nothing reads cu_seqlens on the host), so a training step can
capture them into a CUDA graph and replay it. The test captures forward +
backward once, copies new inputs into the captured buffers, replays, and
compares with the same calls made eagerly on those inputs: O, LSE, dK and dV
bit for bit; dQ bit for bit where it is summed in a fixed order (head_dim
256/512), else within one bf16 rounding (fp32 reductions in arrival order).
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("d128_thd_gqa", "thd", "causal", 3, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300)), {}),
    (Workload("d256_window_chunks", "bshd", "causal", 1, 400, 400, 2, 1, 256, "bf16", window=(100, 0)),
     {"kv_chunk": 128}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_forward_and_backward_replay_from_a_cuda_graph(case):
    import torch

    from parity import gpu_kwargs, to_device
    from scaled_dot_product_02_gb300 import (make_problem, sdpa_bwd, sdpa_bwd_workspace_size, sdpa_fwd,
                                             sdpa_fwd_workspace_size, sdpa_get_device_error)

    w, bwd_kw = case
    first = workloads.make_inputs(w, seed=97)
    second = workloads.make_inputs(w, seed=98)
    kw = gpu_kwargs(w, first)
    if w.layout == "thd":  # the second inputs take the first's lengths (cu_seqlens are captured)
        lens = np.diff(first["cu_seqlens_q"])
        second = workloads.make_inputs(w, seed=98, lengths=lens)
    q, k, v, do = (to_device(first[x], w.dtype) for x in ("q", "k", "v", "do"))
    pb = make_problem(q, k, layout=w.layout, mask=w.mask, window=w.window, scale=w.scale,
                      batch=w.batch if w.layout == "thd" else None, max_seqlen_q=kw.get("max_seqlen_q"),
                      max_seqlen_kv=kw.get("max_seqlen_kv"), **bwd_kw)
    ws_f = torch.empty(max(sdpa_fwd_workspace_size(pb), 256), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(max(sdpa_bwd_workspace_size(pb), 256), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((q.numel() // (q.shape[-1] * q.shape[-2]), q.shape[-2]), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        sdpa_fwd(q, k, v, out=o, lse=lse, workspace=ws_f, **kw)
        sdpa_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws_b, **bwd_kw, **kw)

    # warm up outside the capture (first calls set kernel attributes)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    # replay on new inputs
    for x, name in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
        x.copy_(to_device(second[name], w.dtype))
    graph.replay()
    torch.cuda.synchronize()
    assert sdpa_get_device_error() == 0
    got = [t.clone() for t in (o, lse, dq, dk, dv)]

    # the same calls, eager, on the same inputs
    step()
    torch.cuda.synchronize()
    assert sdpa_get_device_error() == 0
    ref = [o, lse, dq, dk, dv]
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), got, ref):
        if name == "dQ" and w.head_dim == 128:
            diff = (a.float() - b.float()).abs().max().item()
            assert diff <= 2.0 ** -8 * max(1.0, b.float().abs().max().item()), diff
        else:
            assert torch.equal(a, b), f"{name} differs between the graph replay and the eager calls"
