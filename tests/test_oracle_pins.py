"""Pins for the float64 oracle, against things other than the oracle itself.

Each test ties one part of the oracle to something independent of it:
  * library routines: torch's float64 CPU scaled_dot_product_attention with
    its own documented causal masks (upper-left = top-left, lower-right =
    bottom-right), torch.logsumexp, and torch autograd for the gradients;
  * closed forms (zero keys give a uniform average, one key gives that key's
    value, window 0 gives the diagonal value);
  * invariants the pages rely on (top-left and bottom-right coincide when
    Sq == Sk and differ otherwise: TransformerEngine PR #3527,
    "Verification"; GQA equals MHA with repeated KV heads; THD equals the
    per-sequence BSHD runs; SBHD is a transpose of BSHD);
  * central finite differences of L = <dO, O> for every input element.
A plausible slip in the oracle (dropped scale, transposed operand, wrong head
mapping, wrong mask diagonal, wrong gradient sign) fails at least one.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right, causal_upper_left

from oracle import oracle

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _bhsd(x):  # bshd numpy -> (B, H, S, D) torch float64
    return torch.from_numpy(np.ascontiguousarray(x)).permute(0, 2, 1, 3)


def torch_ref(q, k, v, mask, scale, dout=None, gqa=True):
    """Library reference (float64 torch SDPA) on BSHD numpy arrays."""
    qt, kt, vt = (_bhsd(x).clone().requires_grad_(dout is not None) for x in (q, k, v))
    lq, lk = q.shape[1], k.shape[1]
    attn_mask, is_causal = None, False
    if mask == "causal":
        attn_mask = causal_upper_left(lq, lk)._materialize()
    elif mask == "causal_br":
        attn_mask = causal_lower_right(lq, lk)._materialize()
    rep = q.shape[2] // k.shape[2]
    kr = kt.repeat_interleave(rep, dim=1)
    vr = vt.repeat_interleave(rep, dim=1)
    o = F.scaled_dot_product_attention(qt, kr, vr, attn_mask=attn_mask, is_causal=is_causal, scale=scale)
    s = scale * qt @ kr.transpose(-1, -2)
    if attn_mask is not None:
        s = s.masked_fill(~attn_mask, -math.inf)
    lse = torch.logsumexp(s, dim=-1)  # (B, H, S)
    res = {"o": o.permute(0, 2, 1, 3).detach().numpy(),
           "lse": lse.permute(0, 2, 1).reshape(-1, q.shape[2]).detach().numpy()}
    if dout is not None:
        o.backward(_bhsd(dout))
        res["dq"] = qt.grad.permute(0, 2, 1, 3).numpy()
        res["dk"] = kt.grad.permute(0, 2, 1, 3).numpy()
        res["dv"] = vt.grad.permute(0, 2, 1, 3).numpy()
    return res


CASES = [
    # (B, Sq, Sk, Hq, Hkv, D, mask)
    (2, 7, 7, 2, 2, 8, "none"),
    (2, 9, 9, 4, 2, 8, "causal"),
    (1, 6, 11, 4, 1, 4, "causal"),
    (2, 5, 12, 2, 1, 8, "causal_br"),
    (1, 12, 12, 6, 3, 16, "causal_br"),
    (2, 4, 13, 4, 4, 8, "none"),
]


@pytest.mark.parametrize("case", CASES)
def test_forward_and_backward_match_torch_sdpa(case):
    b, sq, sk, hq, hkv, d, mask = case
    r = rng(sum(case[:-1]))
    q, do = r.standard_normal((b, sq, hq, d)), r.standard_normal((b, sq, hq, d))
    k, v = r.standard_normal((b, sk, hkv, d)), r.standard_normal((b, sk, hkv, d))
    scale = 0.37
    ref = torch_ref(q, k, v, mask, scale, dout=do)
    o, lse = oracle.fwd(q, k, v, layout="bshd", mask=mask, scale=scale)
    out = oracle.bwd(q, k, v, do, layout="bshd", mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref["lse"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["o"], ref["o"], rtol=0, atol=1e-12)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(out[key], ref[key], rtol=0, atol=1e-11, err_msg=key)


def test_top_left_equals_bottom_right_when_square_and_differs_when_rectangular():
    r = rng(5)
    q, k, v = r.standard_normal((1, 10, 2, 8)), r.standard_normal((1, 10, 2, 8)), r.standard_normal((1, 10, 2, 8))
    a, la = oracle.fwd(q, k, v, mask="causal")
    b, lb = oracle.fwd(q, k, v, mask="causal_br")
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    k2, v2 = r.standard_normal((1, 16, 2, 8)), r.standard_normal((1, 16, 2, 8))
    a, _ = oracle.fwd(q, k2, v2, mask="causal")
    b, _ = oracle.fwd(q, k2, v2, mask="causal_br")
    assert np.abs(a - b).max() > 1e-3
    # bottom-right: the last query row sees every key, i.e. equals the unmasked row
    c, _ = oracle.fwd(q, k2, v2, mask="none")
    np.testing.assert_allclose(b[:, -1], c[:, -1], atol=1e-13)
    # top-left: the first query row sees only key 0
    np.testing.assert_allclose(a[0, 0], v2[0, 0], atol=1e-13)


def test_zero_keys_give_uniform_average_and_log_count():
    r = rng(6)
    sq = sk = 9
    q, v = r.standard_normal((1, sq, 2, 8)), r.standard_normal((1, sk, 2, 8))
    k = np.zeros_like(v)
    for mask in ("none", "causal"):
        o, lse = oracle.fwd(q, k, v, mask=mask, scale=0.5)
        for i in range(sq):
            n = sk if mask == "none" else i + 1
            np.testing.assert_allclose(o[0, i], v[0, :n].mean(axis=0), atol=1e-13)
            np.testing.assert_allclose(lse[i], [math.log(n)] * 2, atol=1e-13)


def test_single_key_and_dominant_key():
    r = rng(7)
    q, k, v = r.standard_normal((2, 3, 2, 8)), r.standard_normal((2, 1, 2, 8)), r.standard_normal((2, 1, 2, 8))
    o, lse = oracle.fwd(q, k, v, mask="none", scale=0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), atol=1e-14)
    s00 = 0.3 * np.einsum("bshd,bhd->bsh", q, k[:, 0])
    np.testing.assert_allclose(lse, s00.reshape(-1, 2), atol=1e-13)
    # one key far above the rest dominates the softmax
    k2 = np.zeros((1, 5, 1, 4))
    k2[0, 3, 0, 0] = 60.0
    q2 = np.zeros((1, 1, 1, 4))
    q2[0, 0, 0, 0] = 1.0
    v2 = r.standard_normal((1, 5, 1, 4))
    o2, _ = oracle.fwd(q2, k2, v2, mask="none", scale=1.0)
    np.testing.assert_allclose(o2[0, 0, 0], v2[0, 3, 0], atol=1e-20)


def test_diagonal_window_reduces_to_the_identity():
    # causal with a left window of 0: row i sees key i alone, so P = 1, O = V,
    # LSE = the score s_ii, dS = P (dP - delta) = 0 (hence dQ = dK = 0) and dV = dO;
    # with GQA a kv head's dV sums the dO of its query heads
    r = rng(17)
    q, k, v, do = (r.standard_normal(s) for s in [(2, 9, 4, 8), (2, 9, 2, 8), (2, 9, 2, 8), (2, 9, 4, 8)])
    scale = 0.4
    out = oracle.bwd(q, k, v, do, mask="causal", scale=scale, window=(0, 0))
    o, lse = oracle.fwd(q, k, v, mask="causal", scale=scale, window=(0, 0))
    vq = np.repeat(v, 2, axis=2)  # query head h reads kv head h // 2
    np.testing.assert_allclose(o, vq, atol=1e-15)
    s_ii = scale * np.einsum("bshd,bshd->bsh", q, np.repeat(k, 2, axis=2))
    np.testing.assert_allclose(lse, s_ii.reshape(-1, 4), atol=1e-13)
    np.testing.assert_allclose(out["dq"], 0.0, atol=1e-13)
    np.testing.assert_allclose(out["dk"], 0.0, atol=1e-13)
    np.testing.assert_allclose(out["dv"], do.reshape(2, 9, 2, 2, 8).sum(axis=3), atol=1e-13)


def test_lse_rows_of_p_and_delta_identities():
    r = rng(8)
    q, k, v, do = (r.standard_normal(s) for s in [(1, 8, 2, 4), (1, 8, 2, 4), (1, 8, 2, 4), (1, 8, 2, 4)])
    scale = 0.7
    out = oracle.bwd(q, k, v, do, mask="causal", scale=scale)
    # a value vector of ones is reproduced exactly when the rows of P sum to 1
    o1, _ = oracle.fwd(q, k, np.ones_like(v), mask="causal", scale=scale)
    np.testing.assert_allclose(o1, 1.0, atol=1e-14)
    for h in range(2):
        s = scale * q[0, :, h] @ k[0, :, h].T
        s[np.triu_indices(8, 1)] = -np.inf
        lse = np.log(np.exp(s).sum(axis=1))
        np.testing.assert_allclose(out["lse"][:, h], lse, atol=1e-13)
        p = np.exp(s - lse[:, None])
        dp = do[0, :, h] @ v[0, :, h].T
        # delta = rowsum(dO * O) = rowsum(P * dP)
        np.testing.assert_allclose(out["delta"][:, h], (p * dp).sum(axis=1), atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_and_group_sums():
    r = rng(9)
    hq, hkv = 6, 2
    q, do = r.standard_normal((2, 7, hq, 8)), r.standard_normal((2, 7, hq, 8))
    k, v = r.standard_normal((2, 7, hkv, 8)), r.standard_normal((2, 7, hkv, 8))
    kr, vr = np.repeat(k, hq // hkv, axis=2), np.repeat(v, hq // hkv, axis=2)
    g = oracle.bwd(q, k, v, do, mask="causal")
    m = oracle.bwd(q, kr, vr, do, mask="causal")
    np.testing.assert_allclose(g["o"], m["o"], atol=1e-14)
    np.testing.assert_allclose(g["dq"], m["dq"], atol=1e-13)
    np.testing.assert_allclose(g["dk"], m["dk"].reshape(2, 7, hkv, hq // hkv, 8).sum(axis=3), atol=1e-13)
    np.testing.assert_allclose(g["dv"], m["dv"].reshape(2, 7, hkv, hq // hkv, 8).sum(axis=3), atol=1e-13)


@pytest.mark.parametrize("mask", ["none", "causal", "causal_br"])
def test_thd_equals_per_sequence_bshd_and_sbhd_is_transpose(mask):
    r = rng(10)
    lq = np.array([5, 9, 3])
    lk = lq if mask != "causal_br" else np.array([7, 9, 6])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q, do = r.standard_normal((cq[-1], 4, 8)), r.standard_normal((cq[-1], 4, 8))
    k, v = r.standard_normal((ck[-1], 2, 8)), r.standard_normal((ck[-1], 2, 8))
    t = oracle.bwd(q, k, v, do, layout="thd", mask=mask, cu_q=cq, cu_kv=ck)
    for b in range(3):
        sl, kl = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        s = oracle.bwd(q[None, sl], k[None, kl], v[None, kl], do[None, sl], mask=mask)
        np.testing.assert_allclose(t["o"][sl], s["o"][0], atol=1e-14)
        np.testing.assert_allclose(t["lse"][sl], s["lse"], atol=1e-14)
        for key, rs in (("dq", sl), ("dk", kl), ("dv", kl)):
            np.testing.assert_allclose(t[key][rs], s[key][0], atol=1e-13)
    # SBHD: same numbers, rows ordered (s, b)
    qb, kb, vb, dob = (r.standard_normal((2, 6, 2, 8)) for _ in range(4))
    bs = oracle.bwd(qb, kb, vb, dob, layout="bshd", mask=mask)
    tr = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2, 3))
    sb = oracle.bwd(tr(qb), tr(kb), tr(vb), tr(dob), layout="sbhd", mask=mask)
    for key in ("o", "dq", "dk", "dv"):
        np.testing.assert_allclose(sb[key], tr(bs[key]), atol=1e-14)
    np.testing.assert_allclose(sb["lse"], bs["lse"].reshape(2, 6, 2).transpose(1, 0, 2).reshape(12, 2), atol=1e-14)


def test_window_equals_unmasked_attention_over_the_band():
    r = rng(11)
    sq, left = 12, 3
    q, k, v = (r.standard_normal((1, sq, 2, 8)) for _ in range(3))
    o, lse = oracle.fwd(q, k, v, mask="causal", window=(left, 0), scale=0.4)
    for i in range(sq):
        lo = max(0, i - left)
        oi, li = oracle.fwd(q[:, i:i + 1], k[:, lo:i + 1], v[:, lo:i + 1], mask="none", scale=0.4)
        np.testing.assert_allclose(o[:, i], oi[:, 0], atol=1e-14)
        np.testing.assert_allclose(lse[i], li[0], atol=1e-14)
    # a window at least as long as the sequence is plain causal
    o2, _ = oracle.fwd(q, k, v, mask="causal", window=(sq, 0), scale=0.4)
    o3, _ = oracle.fwd(q, k, v, mask="causal", scale=0.4)
    np.testing.assert_array_equal(o2, o3)
    # window 0 keeps only the diagonal
    o4, _ = oracle.fwd(q, k, v, mask="causal", window=(0, 0))
    np.testing.assert_allclose(o4, v, atol=1e-14)
    # bottom-right window: diagonal of row i is i + Sk - Sq
    k5, v5 = r.standard_normal((1, 20, 2, 8)), r.standard_normal((1, 20, 2, 8))
    o5, _ = oracle.fwd(q, k5, v5, mask="causal_br", window=(2, 0), scale=0.4)
    for i in range(sq):
        dg = i + 8
        oi, _ = oracle.fwd(q[:, i:i + 1], k5[:, dg - 2:dg + 1], v5[:, dg - 2:dg + 1], mask="none", scale=0.4)
        np.testing.assert_allclose(o5[:, i], oi[:, 0], atol=1e-14)


def test_fully_masked_rows_are_neutral():
    r = rng(12)
    q, do = r.standard_normal((1, 6, 2, 4)), r.standard_normal((1, 6, 2, 4))
    k, v = r.standard_normal((1, 3, 2, 4)), r.standard_normal((1, 3, 2, 4))
    out = oracle.bwd(q, k, v, do, mask="causal_br")  # rows 0..2 see no key
    assert np.all(out["o"][0, :3] == 0) and np.all(np.isneginf(out["lse"][:3]))
    assert np.all(out["dq"][0, :3] == 0)
    # the remaining rows equal a run without the empty rows
    rest = oracle.bwd(q[:, 3:], k, v, do[:, 3:], mask="causal_br")
    for key in ("dk", "dv"):
        np.testing.assert_allclose(out[key], rest[key], atol=1e-14)


@pytest.mark.parametrize("mask,sq,sk", [("causal", 5, 5), ("causal_br", 3, 6), ("none", 4, 3)])
def test_gradients_match_central_differences(mask, sq, sk):
    r = rng(13 + sq)
    hq, hkv, d = 2, 1, 3
    q, do = r.standard_normal((1, sq, hq, d)), r.standard_normal((1, sq, hq, d))
    k, v = r.standard_normal((1, sk, hkv, d)), r.standard_normal((1, sk, hkv, d))
    scale, eps = 0.8, 1e-6
    g = oracle.bwd(q, k, v, do, mask=mask, scale=scale)

    def loss(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, mask=mask, scale=scale)
        return float(np.sum(o * do))

    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if a is x else a for a in (q, k, v)]
            args_m = [xm if a is x else a for a in (q, k, v)]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_row_samplers_agree_with_full_runs():
    r = rng(14)
    lq = np.array([40, 17])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    q, do = r.standard_normal((cq[-1], 4, 8)), r.standard_normal((cq[-1], 4, 8))
    k, v = r.standard_normal((cq[-1], 2, 8)), r.standard_normal((cq[-1], 2, 8))
    full = oracle.bwd(q, k, v, do, layout="thd", mask="causal", cu_q=cq, cu_kv=cq, window=(5, 0))
    bhi = np.array([[0, 0, 0], [0, 3, 39], [1, 2, 16], [1, 1, 4]])
    o, lse = oracle.fwd_rows(q, k, v, bhi, layout="thd", mask="causal", cu_q=cq, cu_kv=cq, window=(5, 0))
    dq = oracle.dq_rows(q, k, v, do, bhi, layout="thd", mask="causal", cu_q=cq, cu_kv=cq, window=(5, 0))
    for n, (b, h, i) in enumerate(bhi):
        row = cq[b] + i
        np.testing.assert_allclose(o[n], full["o"][row, h], atol=1e-14)
        np.testing.assert_allclose(lse[n], full["lse"][row, h], atol=1e-14)
        np.testing.assert_allclose(dq[n], full["dq"][row, h], atol=1e-14)
    bgj = np.array([[0, 0, 0], [0, 1, 39], [1, 1, 16], [1, 0, 3], [0, 1, 12]])
    dk, dv = oracle.dkdv_rows(q, k, v, do, bgj, layout="thd", mask="causal", cu_q=cq, cu_kv=cq, window=(5, 0))
    for n, (b, g, j) in enumerate(bgj):
        row = cq[b] + j
        np.testing.assert_allclose(dk[n], full["dk"][row, g], atol=1e-14)
        np.testing.assert_allclose(dv[n], full["dv"][row, g], atol=1e-14)
    part = oracle.bwd(q, k, v, do, layout="thd", mask="causal", cu_q=cq, cu_kv=cq, window=(5, 0),
                      batch_range=(1, 2), kv_head_range=(1, 2))
    sl = slice(cq[1], cq[2])
    np.testing.assert_allclose(part["dk"][sl, 1], full["dk"][sl, 1], atol=1e-14)
    np.testing.assert_allclose(part["dq"][sl, 2:], full["dq"][sl, 2:], atol=1e-14)
    assert np.all(part["dk"][sl, 0] == 0) and np.all(part["dk"][: cq[1]] == 0)


# ---------------------------------------------------------------- LSE merge
def _split_keys_forward(q, k, v, bounds, scale):
    """Oracle forward of the queries against each key block [a, b) alone."""
    parts_o, parts_l = [], []
    for a, b in bounds:
        if b > a:
            o, lse = oracle.fwd(q, k[:, a:b], v[:, a:b], layout="bshd", mask="none", scale=scale)
        else:  # an empty block: neutral statistics
            o, lse = np.zeros_like(q), np.full((q.shape[0] * q.shape[1], q.shape[2]), -np.inf)
        parts_o.append(o)
        parts_l.append(lse.reshape(q.shape[0], q.shape[1], q.shape[2]))
    return np.stack(parts_o), np.stack(parts_l)


def test_merge_of_key_blocks_equals_attention_over_all_keys():
    """Attention over the union of key blocks is the log-sum-exp merge of the
    blocks' results; checked against the library reference over all keys,
    with unequal blocks, an empty block and scores large enough that an
    unshifted exp would overflow."""
    r = rng(41)
    q = r.standard_normal((2, 19, 4, 16)) * 10.0  # scores of order 1e3: exp would overflow unshifted
    k = r.standard_normal((2, 70, 2, 16)) * 10.0
    v = r.standard_normal((2, 70, 2, 16))
    scale = 1.3
    po, pl = _split_keys_forward(q, k, v, [(0, 9), (9, 9), (9, 40), (40, 70)], scale)
    o, lse = oracle.merge(po, pl)
    ref = torch_ref(q, k, v, "none", scale)
    assert np.all(np.isfinite(o)) and np.max(ref["lse"]) > 800.0
    np.testing.assert_allclose(o, ref["o"], rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse.reshape(-1, 4), ref["lse"], rtol=1e-14, atol=0)


def test_merge_single_block_is_identity_and_order_does_not_matter():
    r = rng(42)
    po = r.standard_normal((1, 5, 3, 8))
    pl = r.standard_normal((1, 5, 3)) * 3
    o, lse = oracle.merge(po, pl)
    np.testing.assert_array_equal(o, po[0])
    np.testing.assert_array_equal(lse, pl[0])
    po = r.standard_normal((3, 5, 3, 8))
    pl = r.standard_normal((3, 5, 3)) * 3
    perm = [2, 0, 1]
    a = oracle.merge(po, pl)
    b = oracle.merge(po[perm], pl[perm])
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-14)


def test_merge_of_two_equal_blocks_adds_ln2_and_keeps_the_average():
    """Closed form: two blocks with equal LSE weigh one half each."""
    r = rng(43)
    o1, o2 = r.standard_normal((2, 4, 2, 8))
    l0 = r.standard_normal((4, 2))
    o, lse = oracle.merge(np.stack([o1, o2]), np.stack([l0, l0]))
    np.testing.assert_allclose(o, 0.5 * (o1 + o2), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, l0 + math.log(2.0), rtol=0, atol=1e-15)


def test_merge_empty_blocks_are_neutral_and_all_empty_rows_are_zero():
    r = rng(44)
    po = r.standard_normal((3, 6, 2, 8))
    pl = r.standard_normal((3, 6, 2))
    pl[1] = -np.inf               # block 1 saw no keys anywhere
    po[1] = 1.0e30                # whatever it holds must not leak in
    pl[:, 0, :] = -np.inf         # row 0: every block empty
    o, lse = oracle.merge(po, pl)
    keep = oracle.merge(po[[0, 2]], pl[[0, 2]])
    np.testing.assert_allclose(o[1:], keep[0][1:], rtol=0, atol=1e-14)
    assert np.all(o[0] == 0.0) and np.all(lse[0] == -np.inf)


# ------------------------------------------------- asymmetric head dims (d_qk != d_v)
ASYM_CASES = [
    # (B, Sq, Sk, Hq, Hkv, D_qk, D_v, mask)
    (2, 9, 9, 4, 2, 12, 8, "causal"),
    (1, 6, 11, 2, 1, 6, 10, "causal_br"),
    (2, 5, 7, 2, 2, 16, 4, "none"),
]


@pytest.mark.parametrize("case", ASYM_CASES)
def test_asymmetric_head_dims_match_torch_sdpa(case):
    """Library reference: torch's float64 SDPA takes V with its own last
    dimension (E for Q/K, Ev for V); O takes V's width and the LSE is that
    of the Q/K scores."""
    b, sq, sk, hq, hkv, d, dv, mask = case
    r = rng(60 + d + dv)
    q = r.standard_normal((b, sq, hq, d))
    k = r.standard_normal((b, sk, hkv, d))
    v = r.standard_normal((b, sk, hkv, dv))
    ref = torch_ref(q, k, v, mask, 0.29)
    o, lse = oracle.fwd(q, k, v, layout="bshd", mask=mask, scale=0.29)
    assert o.shape == (b, sq, hq, dv)
    np.testing.assert_allclose(o, ref["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref["lse"], rtol=0, atol=1e-12)


def test_asymmetric_value_width_acts_column_by_column_on_thd_and_sbhd():
    """Invariant: each output column is the softmax average of one V column,
    so narrowing V to its first Dv columns narrows O the same way and leaves
    the LSE as it is (compared with the pinned symmetric forward, THD with a
    window and SBHD), and the row sampler follows the full run."""
    r = rng(61)
    lq = np.array([23, 1, 40])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    q = r.standard_normal((cq[-1], 4, 12))
    k = r.standard_normal((cq[-1], 2, 12))
    v_wide = r.standard_normal((cq[-1], 2, 12))
    v = np.ascontiguousarray(v_wide[..., :8])
    kw = dict(layout="thd", mask="causal", cu_q=cq, cu_kv=cq, window=(6, 0), scale=0.4)
    o_w, lse_w = oracle.fwd(q, k, v_wide, **kw)
    o, lse = oracle.fwd(q, k, v, **kw)
    np.testing.assert_allclose(o, o_w[..., :8], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_w, rtol=0, atol=0)
    bhi = np.array([[0, 0, 0], [1, 3, 0], [2, 2, 39], [0, 1, 22]])
    o_r, lse_r = oracle.fwd_rows(q, k, v, bhi, **kw)
    for n, (bb, h, i) in enumerate(bhi):
        np.testing.assert_allclose(o_r[n], o[cq[bb] + i, h], atol=1e-14)
        np.testing.assert_allclose(lse_r[n], lse[cq[bb] + i, h], atol=1e-14)
    qs = r.standard_normal((10, 2, 2, 12))      # SBHD (S, B, H, D)
    ks = r.standard_normal((14, 2, 1, 12))
    vs = r.standard_normal((14, 2, 1, 12))
    o_w, lse_w = oracle.fwd(qs, ks, vs, layout="sbhd", mask="causal_br", scale=0.3)
    o, lse = oracle.fwd(qs, ks, np.ascontiguousarray(vs[..., 5:]), layout="sbhd", mask="causal_br", scale=0.3)
    np.testing.assert_allclose(o, o_w[..., 5:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_w, rtol=0, atol=0)


def test_asymmetric_constant_value_column_comes_back_unchanged():
    """Closed form: the softmax weights of a row sum to one, so a V column
    that holds one constant gives that constant in every row with a key."""
    r = rng(62)
    q = r.standard_normal((1, 12, 2, 16))
    k = r.standard_normal((1, 12, 2, 16))
    v = r.standard_normal((1, 12, 2, 8))
    v[..., 3] = 2.5
    o, _ = oracle.fwd(q, k, v, layout="bshd", mask="causal", scale=0.25)
    np.testing.assert_allclose(o[..., 3], 2.5, rtol=0, atol=1e-14)


def test_backward_rejects_unequal_head_dims():
    r = rng(63)
    q = r.standard_normal((1, 4, 1, 8))
    k = r.standard_normal((1, 4, 1, 8))
    v = r.standard_normal((1, 4, 1, 6))
    with pytest.raises(ValueError):
        oracle.bwd(q, k, v, r.standard_normal((1, 4, 1, 6)), layout="bshd", mask="causal")
    with pytest.raises(ValueError):
        oracle.dq_rows(q, k, v, r.standard_normal((1, 4, 1, 6)), np.array([[0, 0, 1]]), layout="bshd")


# ------------------------------------------------- FP8 E4M3 forward (oracle only)
@pytest.mark.parametrize("case", CASES)
def test_probabilities_match_torch_sdpa_with_identity_values(case):
    """sdpa_oracle_probs against a library routine: torch's float64 SDPA with
    V = the identity over the keys returns P itself (its own causal masks)."""
    b, sq, sk, hq, hkv, d, mask = case
    r = rng(801 + sq)
    q, k = r.standard_normal((b, sq, hq, d)), r.standard_normal((b, sk, hkv, d))
    eye = np.broadcast_to(np.eye(sk)[None, :, None, :], (b, sk, hkv, sk)).copy()
    ref = torch_ref(q, k, eye, mask, 0.4)["o"]  # (B, Sq, Hq, Sk)
    got = oracle.probs(q, k, layout="bshd", mask=mask, scale=0.4).reshape(b, sq, hq, sk)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_probabilities_on_thd_rows_sum_to_one_and_vanish_outside_the_mask():
    r = rng(811)
    cu = np.array([0, 5, 5, 12], dtype=np.int32)
    cuk = np.array([0, 3, 9, 13], dtype=np.int32)
    q, k = r.standard_normal((12, 2, 8)), r.standard_normal((13, 1, 8))
    got = oracle.probs(q, k, layout="thd", mask="causal_br", scale=0.5, cu_q=cu, cu_kv=cuk)
    assert got.shape == (12, 2, 6)
    # sequence 0: 5 queries, 3 keys, bottom-right: query i sees keys <= i - 2
    for i in range(5):
        n = max(0, min(3, i - 1))
        assert np.all(got[i, :, n:] == 0)
        np.testing.assert_allclose(got[i].sum(-1), 1.0 if n else 0.0, rtol=1e-14)
    # sequence 2: 7 queries, 4 keys: rows 0..2 see nothing
    assert np.all(got[5:8] == 0)
    np.testing.assert_allclose(got[8:12].sum(-1), 1.0, rtol=1e-14)


def _e4m3_codes(x):
    """E4M3 codes of float values through torch's own conversion (the library routine)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    np.testing.assert_array_equal(got, ref)                 # NaN codes in the same places
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))  # -0 included; NaN signs carry nothing
    assert np.nanmax(got) == 448.0 and np.nanmin(np.abs(got[got != 0])) == 2.0 ** -9


def test_e4m3_round_matches_torch_and_saturates():
    """Library routine: torch's float8_e4m3fn conversion (round to nearest,
    ties to even) on random values, every grid value and every midpoint
    between neighbours, below the point (464) where torch turns to NaN."""
    r = rng(70)
    grid = np.unique(np.abs(oracle.e4m3_decode(np.arange(256, dtype=np.uint8))))
    grid = grid[np.isfinite(grid)]
    mids = (grid[1:] + grid[:-1]) / 2
    rand = r.uniform(-463.0, 463.0, 20000).astype(np.float32).astype(np.float64)
    tiny = (r.uniform(-1, 1, 5000) * 2.0 ** -6).astype(np.float32).astype(np.float64)
    x = np.concatenate([grid, -grid, mids, -mids, rand, tiny])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_round(x), ref)
    np.testing.assert_array_equal(oracle.e4m3_round(np.array([464.0, 1e6, -500.0])), [448.0, 448.0, -448.0])


def _fp8_inputs(r, shape_q, shape_k, shape_v):
    return (_e4m3_codes(r.standard_normal(s) * 3.0) for s in (shape_q, shape_k, shape_v))


@pytest.mark.parametrize("layout,mask,window", [("bshd", "causal", (-1, -1)), ("thd", "causal_br", (6, -1)),
                                                ("bshd", "none", (-1, -1))])
def test_fp8_scores_and_lse_equal_the_float64_forward_on_decoded_inputs(layout, mask, window):
    """With power-of-two descales the scores are bit for bit those of the
    pinned float64 forward on the decoded, descaled inputs, so the LSE is too;
    O differs only through the E4M3 rounding of P (next test)."""
    r = rng(71)
    dq, dk, dv = 0.5, 0.25, 2.0
    if layout == "thd":
        lens = np.array([17, 30, 1])
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        q8, k8, v8 = _fp8_inputs(r, (cu[-1], 4, 16), (cu[-1], 2, 16), (cu[-1], 2, 16))
        kw = dict(layout="thd", mask=mask, window=window, cu_q=cu, cu_kv=cu, scale=0.3)
    else:
        q8, k8, v8 = _fp8_inputs(r, (2, 12, 4, 16), (2, 19, 2, 16), (2, 19, 2, 16))
        kw = dict(layout="bshd", mask=mask, window=window, scale=0.3)
    o8, l8 = oracle.fwd_fp8(q8, k8, v8, descale=(dq, dk, dv), **kw)
    o, l = oracle.fwd(oracle.e4m3_decode(q8) * dq, oracle.e4m3_decode(k8) * dk, oracle.e4m3_decode(v8) * dv, **kw)
    np.testing.assert_array_equal(l8, l)
    # |dO| <= d_v * max|v| * (2^-4 + n * 2^-10 / 448) per row: one E4M3 rounding of each P * 448
    vmax = np.max(np.abs(oracle.e4m3_decode(v8))) * dv
    n_max = k8.shape[0] if layout == "thd" else k8.shape[1]
    err = np.abs(o8 - o)
    assert np.max(err) <= vmax * (2.0 ** -4 + n_max * 2.0 ** -10 / 448)
    assert np.max(err) > 1e-6 * vmax  # the rounding of P is really applied


def test_fp8_zero_keys_give_the_exact_uniform_average():
    """Closed form: K = 0 makes every allowed score equal, so every
    probability normalised by the row maximum is exp(0) = 1, stored as 448
    exactly, and O is d_v times the mean of the n value rows a row sees, with
    no rounding at all (normalising by the row sum instead would store
    e4m3(448 / n) and miss the mean for most n)."""
    r = rng(72)
    q8 = _e4m3_codes(r.standard_normal((1, 9, 2, 8)))
    k8 = np.zeros((1, 9, 1, 8), dtype=np.uint8)
    v8 = _e4m3_codes(r.standard_normal((1, 9, 1, 8)))
    o, lse = oracle.fwd_fp8(q8, k8, v8, descale=(1.0, 1.0, 0.5), layout="bshd", mask="causal", scale=0.4)
    v = oracle.e4m3_decode(v8)[0, :, 0]
    for i in range(9):
        n = i + 1
        np.testing.assert_allclose(o[0, i, 0], 0.5 * v[:n].mean(axis=0), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(o[0, i, 1], o[0, i, 0], rtol=0, atol=0)   # both q heads read kv head 0
        assert lse[i, 0] == pytest.approx(math.log(n), abs=1e-14)


def test_fp8_stored_probabilities_are_relative_to_the_row_maximum():
    """Two keys with scores s and s - ln 2: normalised by the row maximum the
    stored values are 448 and 224, both exact in E4M3, so O is the weighted
    mean (v0 + v1 / 2) / 1.5 without rounding, whatever the row's scale."""
    q8 = np.zeros((1, 2, 1, 4), dtype=np.uint8)
    k8 = np.zeros((1, 2, 1, 4), dtype=np.uint8)
    q8[..., 0] = _e4m3_codes([1.0])[0]
    k8[0, 0, 0, 0] = _e4m3_codes([2.0])[0]
    k8[0, 1, 0, 0] = _e4m3_codes([1.0])[0]
    v8 = _e4m3_codes(rng(74).standard_normal((1, 2, 1, 4)))
    o, lse = oracle.fwd_fp8(q8, k8, v8, layout="bshd", mask="none", scale=math.log(2.0))
    v = oracle.e4m3_decode(v8)[0, :, 0]
    np.testing.assert_allclose(o[0, 1, 0], (v[0] + 0.5 * v[1]) / 1.5, rtol=1e-15, atol=1e-16)
    assert lse[1, 0] == pytest.approx(2 * math.log(2.0) + math.log(1.5), abs=1e-14)


def test_fp8_dominant_key_returns_its_value_exactly():
    """Closed form: one key scoring far above the rest gets P = 1, stored as
    448 exactly, while the others underflow below E4M3's smallest value, so
    O is that key's value times d_v, bit for bit."""
    q8 = np.zeros((1, 5, 1, 4), dtype=np.uint8)
    k8 = np.zeros((1, 5, 1, 4), dtype=np.uint8)
    q8[..., 0] = _e4m3_codes([448.0])[0]
    k8[0, 0, 0, 0] = _e4m3_codes([448.0])[0]
    v8 = _e4m3_codes(rng(73).standard_normal((1, 5, 1, 4)))
    o, _ = oracle.fwd_fp8(q8, k8, v8, descale=(1.0, 1.0, 0.25), layout="bshd", mask="causal", scale=1.0 / 16)
    v0 = oracle.e4m3_decode(v8)[0, 0, 0] * 0.25
    for i in range(5):
        np.testing.assert_array_equal(o[0, i, 0], v0)
