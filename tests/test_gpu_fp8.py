"""FP8 E4M3 forward (sdpa_fwd_fp8, head_dim 128 and 256) against the float64 oracle.

The kernel follows the oracle's definition step for step (TransformerEngine
PR #3705, closing note on FP8: the softmax output is stored in E4M3 under the
fixed scale 448, normalised by the row's largest probability): S on the
decoded codes, P~ = exp(S - m) against the row's final max m, P8 =
E4M3(P~ * 448) rounded once, O = P8 V * d_v / (448 * l) with l = sum P~.
The two computations of P~ differ only by float32 rounding (relative error
well under 2^-12), so a P8 code can differ from the oracle's only where
P~ * 448 lies within 2^-12 of its value of an E4M3 rounding midpoint, and then
by one E4M3 step. With P~ = p / max_j p (p the oracle's probabilities) and
l = 1 / max_j p, the bound for every element of O is therefore
    (d_v * max p / 448) * sum over those near-midpoint keys of step * |v|
  + (d_v * max p / 448) * 4e-5 * sum_j P8_j |v_j|     (fp32 accumulation)
  + u * |O_ref|            (rounding O to bf16 / fp16: u = 2^-8 / 2^-11)
with the near-midpoint keys found from the oracle's own probabilities, and
LSE within 1e-4. Rows with no allowed key give O = 0 and LSE = -inf exactly.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("fp8_bshd_causal_gqa", "bshd", "causal", 2, 300, 300, 4, 2, 128, "bf16"), None),
    (Workload("fp8_thd_varlen", "thd", "causal", 4, 300, 300, 4, 1, 128, "bf16", len_range=(1, 300)), None),
    (Workload("fp8_sbhd_nomask_fp16", "sbhd", "none", 2, 200, 260, 2, 2, 128, "fp16"), None),
    (Workload("fp8_bottom_right_more_queries", "bshd", "causal_br", 1, 300, 140, 2, 1, 128, "bf16"), None),
    (Workload("fp8_window", "bshd", "causal", 1, 400, 400, 2, 2, 128, "bf16", window=(100, 0)), None),
    (Workload("fp8_thd_unequal_bottom_right", "thd", "causal_br", 5, 300, 333, 4, 2, 128, "bf16"),
     ([300, 1, 129, 200, 64], [140, 250, 129, 333, 1])),
    # head_dim 256 (one query-tile pipeline per CTA)
    (Workload("fp8_d256_bshd_causal_gqa", "bshd", "causal", 2, 300, 300, 4, 2, 256, "bf16"), None),
    (Workload("fp8_d256_thd_varlen", "thd", "causal", 4, 300, 300, 4, 1, 256, "bf16", len_range=(1, 300)), None),
    (Workload("fp8_d256_sbhd_window_fp16", "sbhd", "causal", 2, 400, 400, 2, 2, 256, "fp16", window=(100, 0)), None),
    (Workload("fp8_d256_bottom_right_nomask_rect", "bshd", "none", 1, 200, 333, 2, 1, 256, "bf16"), None),
    (Workload("fp8_two_sided_window", "bshd", "none", 1, 300, 300, 2, 2, 128, "bf16", window=(70, 45)), None),
    (Workload("fp8_d256_br_window", "bshd", "causal_br", 1, 200, 333, 2, 1, 256, "bf16", window=(90, 0)), None),
    # every row sees only its own key: each query tile has one key tile, so at
    # head_dim 256 one softmax warpgroup has no pass-1 step and the other no
    # pass-2 step, tile after tile
    (Workload("fp8_diagonal_window", "bshd", "causal", 2, 600, 600, 4, 2, 128, "bf16", window=(0, 0)), None),
    (Workload("fp8_d256_diagonal_window", "bshd", "causal", 2, 600, 600, 4, 2, 256, "bf16", window=(0, 0)), None),
    # empty sequences between live ones
    (Workload("fp8_thd_with_empty", "thd", "causal", 5, 150, 150, 4, 2, 128, "bf16"),
     ([150, 0, 37, 0, 90], [150, 0, 37, 0, 90])),
    (Workload("fp8_d256_thd_with_empty_br", "thd", "causal_br", 4, 120, 200, 2, 1, 256, "bf16"),
     ([0, 120, 0, 33], [0, 200, 0, 33])),
]
UNIT = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}  # unit roundoff of the output format


def _e4m3_step(x):
    """Distance between adjacent E4M3 values around x >= 0 (2^-9 among the
    subnormals, 2^(e-3) in [2^e, 2^(e+1)))."""
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -30)))
    return 2.0 ** (np.maximum(e, -6.0) - 3.0)


def _kv_rows(w, inp, b):
    if w.layout == "thd":
        return slice(int(inp["cu_seqlens_kv"][b]), int(inp["cu_seqlens_kv"][b + 1]))
    return b


def _q_rows(w, inp, b):
    """Token rows of sequence b's queries, in order."""
    if w.layout == "thd":
        return np.arange(int(inp["cu_seqlens_q"][b]), int(inp["cu_seqlens_q"][b + 1]))
    if w.layout == "bshd":
        return b * w.seqlen_q + np.arange(w.seqlen_q)
    return np.arange(w.seqlen_q) * w.batch + b


def _bound(w, inp, probs, o_ref, v):
    """Elementwise bound on |O - O_ref| (see the module docstring)."""
    dvs = workloads.FP8_DESCALE[2]
    pmax = probs.max(axis=-1, keepdims=True)  # the row's largest probability (0 for rows without keys)
    x = np.divide(probs, pmax, out=np.zeros_like(probs), where=pmax > 0) * 448.0
    step = _e4m3_step(x)
    frac = x / step - np.floor(x / step)
    near = (np.abs(frac - 0.5) * step <= 2.0 ** -12 * x) & (x > 0)
    tie_w = np.where(near, step, 0.0) * pmax  # the division by l = 1 / max p
    acc_w = x * 4e-5 * pmax
    o_flat = o_ref.reshape(-1, w.heads_q, w.head_dim)
    bound = np.zeros_like(o_flat)
    group = w.heads_q // w.heads_kv
    nb = len(inp["cu_seqlens_q"]) - 1 if w.layout == "thd" else w.batch
    for b in range(nb):
        rows = _q_rows(w, inp, b)
        if w.layout == "sbhd":
            vb = np.abs(v[:, b])  # (Sk, Hkv, 128)
        else:
            vb = np.abs(v[_kv_rows(w, inp, b)])
        lk = vb.shape[0]
        for h in range(w.heads_q):
            vh = vb[:, h // group, :]
            bound[rows, h] = (tie_w[rows, h, :lk] @ vh) * (1 + 2.0 ** -8) + acc_w[rows, h, :lk] @ vh
    bound *= dvs / 448.0
    return bound + UNIT[w.dtype] * np.abs(o_flat) + 1e-7


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_fp8_forward_matches_oracle(case):
    import torch

    from oracle import oracle
    from parity import gpu_kwargs
    from scaled_dot_product_02_gb300 import sdpa_fwd_fp8, sdpa_get_device_error

    w, lens = case
    inp = workloads.fp8_inputs(w, seed=61, lengths=None if lens is None else tuple(np.array(x) for x in lens))
    kw = gpu_kwargs(w, inp)
    q8, k8, v8 = (torch.from_numpy(inp[x]).cuda() for x in ("q8", "k8", "v8"))
    out_dtype = {"bf16": torch.bfloat16, "fp16": torch.float16}[w.dtype]
    o, lse = sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, out_dtype=out_dtype, **kw)
    assert sdpa_get_device_error() == 0
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)

    okw = dict(layout=w.layout, mask=w.mask, scale=w.scale, window=w.window)
    if w.layout == "thd":
        okw.update(cu_q=inp["cu_seqlens_q"], cu_kv=inp["cu_seqlens_kv"])
    o_ref, l_ref = oracle.fwd_fp8(inp["q8"], inp["k8"], inp["v8"], descale=workloads.FP8_DESCALE, **okw)
    dq, dk, dv = workloads.FP8_DESCALE
    qd, kd, vd = (oracle.e4m3_decode(inp[x]) for x in ("q8", "k8", "v8"))
    probs = oracle.probs(qd * dq, kd * dk, **okw)
    bound = _bound(w, inp, probs, o_ref, vd).reshape(o.shape)

    empty = np.isneginf(l_ref)
    assert np.all(np.isneginf(lse[empty])), "rows without keys must have LSE = -inf"
    assert np.all(o.reshape(-1, w.heads_q, w.head_dim)[empty] == 0), "rows without keys must have O = 0"
    with np.errstate(invalid="ignore"):
        lse_err = float(np.max(np.abs(np.where(empty, 0.0, lse - l_ref))))
    excess = np.abs(o - o_ref) / bound
    worst = float(np.max(excess))
    print(f"[{w.name}] O: max|O-O_ref|={np.max(np.abs(o - o_ref)):.3e} worst err/bound={worst:.3f} "
          f"median bound={np.median(bound):.3e}; LSE err={lse_err:.3e} ({int(empty.sum())} empty rows)")
    assert lse_err <= 1e-4
    assert worst <= 1.0, f"O exceeds its bound by {worst:.2f}x"


FULL = [workloads.VARLEN_THD, workloads.LONG_FP16, workloads.SLIDING]


@pytest.mark.slow
@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_fp8_full_size_sampled_rows(w):
    """The FP8 forward at the full workload shapes, in the configuration the
    benchmark times (bf16 O), checked on sampled query rows. Under top-left
    causal, row i of a sequence sees exactly its keys 0..i (max(0, i - w) ..
    i under a left window w), so the oracle checks each sampled row as a
    one-query problem over those keys with no mask, under the same bound as
    the small cases."""
    import torch

    from oracle import oracle
    from parity import gpu_kwargs, kv_token_row, sample_rows, token_row
    from scaled_dot_product_02_gb300 import sdpa_fwd_fp8, sdpa_get_device_error

    assert w.mask == "causal" and w.window[1] in (-1, 0) and w.head_dim in (128, 256)
    D = w.head_dim
    inp = workloads.fp8_inputs(w)
    kw = gpu_kwargs(w, inp)
    q8, k8, v8 = (torch.from_numpy(inp[x]).cuda() for x in ("q8", "k8", "v8"))
    o, lse = sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, out_dtype=torch.bfloat16, **kw)
    assert sdpa_get_device_error() == 0
    o = o.float().cpu().numpy().astype(np.float64).reshape(-1, w.heads_q, D)
    lse = lse.cpu().numpy().astype(np.float64).reshape(-1, w.heads_q)
    del q8, k8, v8
    torch.cuda.empty_cache()

    group = w.heads_q // w.heads_kv
    qs, ks, vs = (inp[x].reshape(-1, n, D) for x, n in (("q8", w.heads_q), ("k8", w.heads_kv), ("v8", w.heads_kv)))
    dq, dk, _ = workloads.FP8_DESCALE
    okw = dict(layout="bshd", mask="none", scale=w.scale)
    worst, lse_err = 0.0, 0.0
    rows = sample_rows(w, inp, 40, seed=17)
    for b, h, i in rows:
        t = token_row(w, inp, int(b), int(i))
        j0 = max(0, int(i) - w.window[0]) if w.window[0] >= 0 else 0
        kv = np.array([kv_token_row(w, inp, int(b), j) for j in range(j0, int(i) + 1)])
        sub = {"q8": qs[t, h][None, None, None, :], "k8": ks[kv, h // group][None, :, None, :],
               "v8": vs[kv, h // group][None, :, None, :]}
        sw = Workload("row", "bshd", "none", 1, 1, len(kv), 1, 1, D, "bf16")
        o_ref, l_ref = oracle.fwd_fp8(sub["q8"], sub["k8"], sub["v8"], descale=workloads.FP8_DESCALE, **okw)
        probs = oracle.probs(oracle.e4m3_decode(sub["q8"]) * dq, oracle.e4m3_decode(sub["k8"]) * dk, **okw)
        bound = _bound(sw, sub, probs, o_ref, oracle.e4m3_decode(sub["v8"])).reshape(D)
        worst = max(worst, float(np.max(np.abs(o[t, h] - o_ref.reshape(D)) / bound)))
        lse_err = max(lse_err, abs(float(lse[t, h]) - float(np.ravel(l_ref)[0])))
    print(f"[{w.name} fp8, {len(rows)} sampled rows] worst err/bound={worst:.3f}; LSE err={lse_err:.3e}")
    assert lse_err <= 1e-4
    assert worst <= 1.0, f"O exceeds its bound by {worst:.2f}x"
