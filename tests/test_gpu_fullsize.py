"""Full-size parity: every workload at its real shape, through the same calls
the benchmark times, checked on sampled rows that the float64 oracle computes
one by one (query rows for O/LSE/dQ; key rows of one (sequence, kv head) for
dK/dV), under the same per-case floor rule as the small cases. Forward-only
workloads (asymmetric head dims) check O and LSE."""
import numpy as np
import pytest

import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def run_full(w, inp):
    import torch

    from parity import gpu_kwargs, to_device, report
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    if w.name in workloads.FORWARD_ONLY:
        assert sdpa_get_device_error() == 0
        out = {"o": f(o), "lse": lse.cpu().numpy().astype(np.float64)}
        del q, k, v, do, o, lse
        torch.cuda.empty_cache()
        return out
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, **kw)
    assert sdpa_get_device_error() == 0
    out = {"o": f(o), "lse": lse.cpu().numpy().astype(np.float64), "dq": f(dq), "dk": f(dk), "dv": f(dv)}
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    return out


@pytest.mark.parametrize("w", workloads.ALL, ids=lambda w: w.name)
def test_full_size_sampled_parity(w):
    from parity import check_bwd, check_fwd, check_sampled, report

    inp = workloads.make_inputs(w)
    out = run_full(w, inp)
    if w.name in workloads.FORWARD_ONLY:
        results = check_sampled(w, inp, out, n_rows=48, backward=False)
    elif w.batch * w.seqlen_q * w.heads_q <= 4096:
        # small enough for the oracle to check every element
        results = check_fwd(w, inp, out["o"], out["lse"]) + check_bwd(w, inp, out["dq"], out["dk"], out["dv"])
    else:
        results = check_sampled(w, inp, out, n_rows=48, n_keys=24)
    report(w.name, results)
