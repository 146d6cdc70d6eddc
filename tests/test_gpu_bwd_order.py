"""The sequence order of the head_dim 128 THD backward.

The THD metadata guard (TransformerEngine PR #3705, "Execution and supported
scope": the cumulative lengths are checked on the GPU on every execution)
also writes the order in which the backward grid takes the sequences: their
indices by query-tile count, longest first. The order only decides when a
sequence's CTAs start; these tests check that it is a permutation sorted as
stated (read from the backward's workspace, where it sits after the guard
word) and that a backward over many sequences of mixed lengths, empty ones
included, still matches the float64 oracle.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

ORDER_OFFSET = 256  # bytes: after the guard word's block


def _lengths(n, hi, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, hi + 1, size=n)
    lens[::17] = 0
    lens[5] = hi
    return lens


@pytest.mark.parametrize("n_seq,hi", [(7, 700), (300, 150)])
def test_guard_orders_sequences_longest_first(n_seq, hi):
    import torch

    from parity import check_bwd, gpu_kwargs, report, to_device
    from scaled_dot_product_02_gb300 import (make_problem, sdpa_bwd, sdpa_bwd_workspace_size, sdpa_fwd,
                                             sdpa_get_device_error)

    lens = _lengths(n_seq, hi, seed=n_seq)
    w = Workload(f"order_{n_seq}", "thd", "causal", n_seq, int(lens.max()), int(lens.max()), 4, 2, 128, "bf16")
    inp = workloads.make_inputs(w, seed=31, lengths=lens)
    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    p = make_problem(q, k, layout="thd", mask="causal", scale=w.scale, batch=n_seq, max_seqlen_q=kw["max_seqlen_q"],
                     max_seqlen_kv=kw["max_seqlen_kv"])
    ws = torch.zeros(sdpa_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert sdpa_get_device_error() == 0

    order = ws[ORDER_OFFSET:ORDER_OFFSET + 4 * n_seq].cpu().view(torch.int32).numpy()
    assert sorted(order.tolist()) == list(range(n_seq)), "not a permutation of the sequences"
    tiles = -(-lens[order] // 64)
    assert np.all(np.diff(tiles) <= 0), f"query-tile counts along the order: {tiles.tolist()}"

    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    report(w.name, check_bwd(w, inp, f(dq), f(dk), f(dv)))
