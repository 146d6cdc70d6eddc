"""GPU parity of the asymmetric forward: Q and K rows of 192 entries, V and O
rows of 128 (TransformerEngine PR #3527, "Scope": the forward prefill engine
lists (192, 128) among its native head-dim pairs; the backward there, and
here, requires d_qk == d_v).

Every case compares O and LSE with the float64 oracle element by element
under the same per-case floor rule as the symmetric forward, across layouts,
masks, windows, GQA, ragged tiles and empty rows; the backward declines the
pair with SDPA_ERR_UNSUPPORTED.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu


def W(name, layout, mask, b, sq, sk, hq, hkv, dtype="bf16", **kw):
    return Workload(name, layout, mask, b, sq, sk, hq, hkv, 192, dtype, head_dim_v=128, **kw)


CASES = [
    W("bshd_causal_gqa_ragged", "bshd", "causal", 2, 300, 300, 4, 2),
    W("sbhd_fp16_nomask", "sbhd", "none", 2, 200, 200, 2, 2, "fp16", std=0.5),
    W("thd_varlen_gqa", "thd", "causal", 4, 300, 300, 4, 1, len_range=(1, 300)),
    W("bottom_right_rect", "bshd", "causal_br", 1, 200, 333, 2, 1),
    W("br_more_queries_than_keys", "bshd", "causal_br", 1, 300, 140, 2, 2),
    W("sliding_window", "bshd", "causal", 1, 400, 400, 2, 2, window=(100, 0)),
    W("two_sided_window", "bshd", "none", 1, 300, 300, 2, 2, window=(20, 37)),
    W("one_query", "bshd", "none", 2, 1, 200, 2, 1),
    W("one_key", "bshd", "causal_br", 1, 130, 1, 2, 2),
    W("tiny_thd_sequences", "thd", "causal", 40, 3, 3, 2, 1, len_range=(1, 3)),
    W("gqa_16_to_1_fp16", "bshd", "causal", 1, 256, 256, 16, 1, "fp16"),
    W("diagonal_window", "bshd", "causal", 1, 300, 300, 2, 2, window=(0, 0)),  # every row sees its own key alone
]


def _fwd(w, inp):
    from parity import gpu_kwargs, to_device, report
    from scaled_dot_product_02_gb300 import sdpa_fwd, sdpa_get_device_error

    q, k, v = (to_device(inp[x], w.dtype) for x in ("q", "k", "v"))
    o, lse = sdpa_fwd(q, k, v, **gpu_kwargs(w, inp))
    assert sdpa_get_device_error() == 0
    assert o.shape == q.shape[:-1] + (128,)
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_asymmetric_forward_matches_oracle(w):
    from parity import check_fwd, report

    inp = workloads.make_inputs(w, seed=31)
    o, lse = _fwd(w, inp)
    results = check_fwd(w, inp, o, lse)
    report(w.name, results)


def test_asymmetric_forward_with_empty_thd_sequences():
    from parity import check_fwd, report

    w = W("thd_with_empty", "thd", "causal", 4, 150, 150, 2, 2)
    inp = workloads.make_inputs(w, seed=32, lengths=np.array([150, 0, 37, 0]))
    o, lse = _fwd(w, inp)
    results = check_fwd(w, inp, o, lse)
    report(w.name, results)


@pytest.mark.parametrize("mask", ["causal_br", "causal", "none"])
def test_asymmetric_forward_with_unequal_thd_lengths(mask):
    # per-sequence query and key lengths differ (cu_seqlens_q != cu_seqlens_kv): a
    # sequence with more queries than keys (its first rows see no key under the
    # bottom-right mask), one with a single query, equal lengths, fewer queries than
    # keys and a single key
    from parity import check_fwd, report

    lq, lk = [300, 1, 129, 200, 64], [140, 250, 129, 333, 1]
    w = W(f"thd_unequal_{mask}", "thd", mask, len(lq), max(lq), max(lk), 4, 2)
    inp = workloads.make_inputs(w, seed=41, lengths=(np.array(lq), np.array(lk)))
    assert not np.array_equal(inp["cu_seqlens_q"], inp["cu_seqlens_kv"])
    o, lse = _fwd(w, inp)
    results = check_fwd(w, inp, o, lse)
    report(w.name, results)


def test_asymmetric_backward_is_declined():
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    q = torch.randn(1, 128, 2, 192, device="cuda", dtype=torch.bfloat16)
    k = torch.randn_like(q)
    v = torch.randn(1, 128, 2, 128, device="cuda", dtype=torch.bfloat16)
    o, lse = sdpa.sdpa_fwd(q, k, v, mask="causal")
    assert sdpa.sdpa_get_device_error() == 0
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_bwd(q, k, v, o, lse, torch.randn_like(o), mask="causal")
    assert e.value.status == 2  # SDPA_ERR_UNSUPPORTED
