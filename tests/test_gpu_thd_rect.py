"""Compact THD with different query and key lengths per sequence
(cu_seqlens_q != cu_seqlens_kv; TransformerEngine PR #3705, "Execution and
supported scope": per-sequence cumulative lengths for Q and for KV), forward
and backward against the float64 oracle under the per-case floor rule.

Per sequence b the bottom-right diagonal of query i is key i + Lk_b - Lq_b
(PR #3527, "Verification": rectangular bottom-right cases), so the lengths
mix Lq_b > Lk_b (bottom-right: the first Lq_b - Lk_b rows see no key and
must come back as O = 0, LSE = -inf, dQ = 0), Lq_b < Lk_b, equal lengths, a
single query and a single key, at head_dim 128, 256 and 512, with GQA (up to
8:1), windows, and empty sequences between live ones.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

LENS_Q = [300, 1, 129, 200, 64]
LENS_KV = [140, 250, 129, 333, 1]


def _case(name, mask, d, heads=(4, 2), dtype="bf16", window=(-1, -1), lens=(LENS_Q, LENS_KV)):
    lq, lk = lens
    w = Workload(name, "thd", mask, len(lq), max(lq), max(lk), heads[0], heads[1], d, dtype, window=window)
    return w, (np.array(lq), np.array(lk))


CASES = [
    _case("d128_bottom_right", "causal_br", 128),
    _case("d128_top_left", "causal", 128),
    _case("d128_nomask", "none", 128),
    _case("d128_bottom_right_window", "causal_br", 128, window=(64, 0)),
    _case("d128_fp16_bottom_right", "causal_br", 128, dtype="fp16"),
    _case("d256_bottom_right", "causal_br", 256),
    _case("d256_top_left", "causal", 256, heads=(2, 1)),
    _case("d512_bottom_right", "causal_br", 512, heads=(2, 1)),
    _case("d512_top_left", "causal", 512, heads=(2, 2)),
    _case("d512_nomask_fp16", "none", 512, heads=(2, 1), dtype="fp16"),
    _case("d256_top_left_window", "causal", 256, window=(100, 0)),
    _case("d512_bottom_right_window", "causal_br", 512, heads=(2, 1), window=(80, 0)),
    _case("d128_gqa_8_to_1", "causal", 128, heads=(8, 1)),
    # empty sequences (no query and no key) between live ones
    _case("d256_with_empty", "causal", 256, heads=(2, 1), lens=([150, 0, 37, 0, 90], [150, 0, 60, 0, 90])),
    _case("d512_with_empty_br", "causal_br", 512, heads=(2, 2), lens=([0, 120, 0, 33], [0, 200, 0, 33])),
]


def _run(w, inp, deterministic=False):
    from parity import gpu_kwargs, to_device, report
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, deterministic=deterministic, **kw)
    assert sdpa_get_device_error() == 0
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f(o), lse.cpu().numpy().astype(np.float64), f(dq), f(dk), f(dv)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_thd_unequal_lengths_match_oracle(case):
    from parity import check_bwd, check_fwd, report

    w, lens = case
    inp = workloads.make_inputs(w, seed=23, lengths=lens)
    assert not np.array_equal(inp["cu_seqlens_q"], inp["cu_seqlens_kv"])
    o, lse, dq, dk, dv = _run(w, inp)
    res = check_fwd(w, inp, o, lse) + check_bwd(w, inp, dq, dk, dv)
    report(w.name, res)
    if w.mask == "causal_br" and lens[0][0] == 300 and lens[1][0] == 140:
        # sequence 0: Lq 300 > Lk 140, so its first 160 rows see no key
        a = int(inp["cu_seqlens_q"][0])
        assert np.all(np.isneginf(lse[a:a + 160])) and np.all(o[a:a + 160] == 0) and np.all(dq[a:a + 160] == 0)


def test_thd_unequal_lengths_deterministic_backward():
    from parity import check_bwd, check_fwd, report

    w, lens = _case("d128_bottom_right_det", "causal_br", 128)
    inp = workloads.make_inputs(w, seed=29, lengths=lens)
    o, lse, dq, dk, dv = _run(w, inp, deterministic=True)
    res = check_fwd(w, inp, o, lse) + check_bwd(w, inp, dq, dk, dv)
    report(w.name, res)
