"""The benchmark's FLOP accounting against the oracle's mask semantics (CPU).

bench.py counts unmasked (query, key) pairs in closed form per row to turn
kernel times into TFLOP/s. With K = 0 every allowed score is 0, so the
oracle's LSE of a row is ln(number of keys it may attend) (a closed form the
oracle pins hold); summing exp(LSE) over rows therefore counts the pairs the
oracle's own mask allows, independently of the benchmark's formula.
tests/golden/pair_counts.json holds those counts for every workload at full
size (written by tests/golden/make_pair_counts.py, which calls only the
oracle); the benchmark's counts and the closed forms of the masks must both
reproduce them.
"""
import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402
from oracle import oracle  # noqa: E402

SHAPES = [
    # (Sq, Sk, mask, window)
    (37, 37, "none", (-1, -1)),
    (37, 37, "causal", (-1, -1)),
    (20, 53, "causal", (-1, -1)),
    (53, 20, "causal", (-1, -1)),
    (20, 53, "causal_br", (-1, -1)),
    (53, 20, "causal_br", (-1, -1)),
    (64, 64, "causal", (9, -1)),
    (30, 70, "causal_br", (5, -1)),
    (48, 48, "none", (7, 11)),
    (48, 48, "none", (0, 0)),
]


def oracle_pairs(sq, sk, mask, window):
    """Pairs the oracle's mask allows for one head: sum over rows of exp(LSE) with K = 0."""
    q = np.ones((1, sq, 1, 4))
    k = np.zeros((1, sk, 1, 4))
    v = np.zeros((1, sk, 1, 4))
    _, lse = oracle.fwd(q, k, v, layout="bshd", mask=mask, scale=1.0, window=window)
    finite = np.isfinite(lse)
    return int(round(float(np.sum(np.exp(lse[finite])))))


@pytest.mark.parametrize("sq,sk,mask,window", SHAPES)
def test_pair_count_matches_the_oracle_mask(sq, sk, mask, window):
    w = workloads.Workload("acct", "bshd", mask, 1, sq, sk, 1, 1, 128, "bf16", window=window)
    assert bench.pairs_per_head(w, sq, sk) == oracle_pairs(sq, sk, mask, window)


def test_flops_use_both_head_dims_and_the_causal_convention():
    lens = np.array([100, 37, 0, 64])
    inp = {"cu_seqlens_q": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)}
    inp["cu_seqlens_kv"] = inp["cu_seqlens_q"]
    w = workloads.Workload("acct_thd", "thd", "causal", 4, 100, 100, 8, 2, 192, "bf16", head_dim_v=128)
    conv, exact = bench.flops(w, inp)
    per_pair = 2 * 192 + 2 * 128
    assert conv == sum(per_pair * 8 * int(n) * int(n) // 2 for n in lens)
    assert exact == sum(per_pair * 8 * int(n) * (int(n) + 1) // 2 for n in lens)  # causal: n(n+1)/2 pairs
    # equal head dims reduce to 4 * D per pair
    w2 = w.replace(head_dim=128, head_dim_v=0)
    assert bench.flops(w2, inp)[1] == sum(4 * 128 * 8 * int(n) * (int(n) + 1) // 2 for n in lens)


def test_headline_workload_flops_are_the_stated_convention():
    w = workloads.VARLEN_THD
    lq = workloads.thd_lengths(w)
    assert list(lq) == [3750, 2708, 3452, 568, 2333, 1184, 3263, 3587]  # the lengths the bench line reports
    inp = {"cu_seqlens_q": np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)}
    inp["cu_seqlens_kv"] = inp["cu_seqlens_q"]
    conv, exact = bench.flops(w, inp)
    assert conv == sum(4 * w.heads_q * int(n) * int(n) * w.head_dim // 2 for n in lq)
    # the exact count adds the diagonal: n(n+1)/2 against n^2/2 pairs
    assert math.isclose(exact / conv, sum(int(n) * (int(n) + 1) for n in lq) / sum(int(n) ** 2 for n in lq))


def _golden():
    import json

    with open(os.path.join(ROOT, "tests", "golden", "pair_counts.json")) as f:
        return json.load(f)["workloads"]


def _closed_form(sq, sk, mask, window):
    """Pairs per head from the mask definition, summed in closed form."""
    wl = window[0]
    if mask == "none" and wl < 0:
        return sq * sk
    if mask == "causal" and wl < 0 and sq == sk:
        return sq * (sq + 1) // 2
    if mask == "causal" and sq == sk:             # a left window of wl keys beyond the diagonal
        full = min(sq, wl + 1)
        return full * (full + 1) // 2 + (sq - full) * (wl + 1)
    if mask == "causal_br" and wl < 0 and sq <= sk:  # row i sees i + (sk - sq) + 1 keys
        return sq * (sk - sq) + sq * (sq + 1) // 2
    raise ValueError("no closed form for this shape")


@pytest.mark.parametrize("w", workloads.ALL, ids=lambda w: w.name)
def test_pair_counts_of_every_workload_match_the_golden_oracle_counts(w):
    g = _golden()[w.name]
    if w.layout == "thd":
        lens = workloads.thd_lengths(w)
        assert list(lens) == g["lengths"]
        for n, want in zip(lens, g["pairs_per_sequence"]):
            assert bench.pairs_per_head(w, int(n), int(n)) == want == _closed_form(int(n), int(n), w.mask, w.window)
    else:
        want = g["pairs"]
        assert bench.pairs_per_head(w, w.seqlen_q, w.seqlen_kv) == want
        assert _closed_form(w.seqlen_q, w.seqlen_kv, w.mask, w.window) == want
