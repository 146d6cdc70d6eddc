"""Exactness of masks and varlen boundaries: bitwise properties, not
tolerances (the spec requirement that masks and varlen boundaries be
exact, read as four checks):

(i)   K/V rows that a query may not attend (keys past its causal diagonal,
      keys no query sees, another sequence's rows) do not change its O or LSE
      in any bit;
(ii)  keys that no query attends get dK = dV = 0 exactly;
(iii) a THD call gives, sequence by sequence, bit for bit the results of a
      batch-1 BSHD call on that sequence alone (forward, and the
      deterministic backward);
(iv)  nothing past the outputs' rows is written (canaries after the buffers).

Every input is seeded; the kernels are the ones the parity tests check.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

DIMS = [(128, 128), (256, 256), (512, 512), (192, 128)]  # (head_dim, head_dim_v)


def _randn(gen, *shape, scale=1.0):
    import torch

    return (torch.randn(*shape, generator=gen, device="cuda") * scale).to(torch.bfloat16)


def _gen(seed):
    import torch

    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


@pytest.mark.parametrize("d,dv", DIMS, ids=lambda x: str(x))
def test_keys_a_row_may_not_attend_leave_its_output_unchanged(d, dv):
    import torch

    from scaled_dot_product_02_gb300 import sdpa_fwd, sdpa_get_device_error

    g = _gen(d + dv)
    # top-left causal, Sq 200 < Sk 333: keys 200.. are seen by no query, and
    # key 150 only by rows 150.. (inside the second key tile, an edge tile)
    q = _randn(g, 1, 200, 4, d)
    k = _randn(g, 1, 333, 2, d)
    v = _randn(g, 1, 333, 2, dv)
    o1, l1 = sdpa_fwd(q, k, v, mask="causal")
    k2, v2 = k.clone(), v.clone()
    k2[:, 200:] = _randn(g, 1, 133, 2, d, scale=8.0)
    v2[:, 200:] = _randn(g, 1, 133, 2, dv, scale=8.0)
    o2, l2 = sdpa_fwd(q, k2, v2, mask="causal")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    k2[:, 150] = _randn(g, 1, 2, d, scale=8.0)
    v2[:, 150] = _randn(g, 1, 2, dv, scale=8.0)
    o3, l3 = sdpa_fwd(q, k2, v2, mask="causal")
    assert sdpa_get_device_error() == 0
    assert torch.equal(o3[:, :150], o1[:, :150]) and torch.equal(l3[:150], l1[:150])
    assert not torch.equal(o3[:, 150:], o1[:, 150:])  # the rows that see key 150 do change


@pytest.mark.parametrize("d,dv", DIMS, ids=lambda x: str(x))
def test_other_sequences_rows_leave_a_thd_sequence_unchanged(d, dv):
    import torch

    from scaled_dot_product_02_gb300 import sdpa_fwd, sdpa_get_device_error

    g = _gen(7 * d + dv)
    lens = [200, 150, 77]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    t = sum(lens)
    q = _randn(g, t, 4, d)
    k = _randn(g, t, 2, d)
    v = _randn(g, t, 2, dv)
    kw = dict(layout="thd", mask="causal", cu_seqlens_q=cu, cu_seqlens_kv=cu, max_seqlen_q=200, max_seqlen_kv=200)
    o1, l1 = sdpa_fwd(q, k, v, **kw)
    k2, v2 = k.clone(), v.clone()
    k2[200:350] = _randn(g, 150, 2, d, scale=8.0)  # sequence 1's keys and values
    v2[200:350] = _randn(g, 150, 2, dv, scale=8.0)
    o2, l2 = sdpa_fwd(q, k2, v2, **kw)
    assert sdpa_get_device_error() == 0
    for a, b in ((0, 200), (350, 427)):
        assert torch.equal(o1[a:b], o2[a:b]) and torch.equal(l1[a:b], l2[a:b])
    assert not torch.equal(o1[200:350], o2[200:350])


@pytest.mark.parametrize("d,deterministic", [(128, False), (128, True), (256, False), (512, False)])
def test_keys_no_query_attends_get_zero_gradients(d, deterministic):
    import torch

    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    g = _gen(d + int(deterministic))
    q = _randn(g, 1, 200, 4, d)
    k = _randn(g, 1, 333, 2, d)
    v = _randn(g, 1, 333, 2, d)
    do = _randn(g, 1, 200, 4, d)
    o, lse = sdpa_fwd(q, k, v, mask="causal")
    dq, dk, dv = sdpa_bwd(q, k, v, o, lse, do, mask="causal", deterministic=deterministic)
    assert sdpa_get_device_error() == 0
    # keys 200..332 are past every query's diagonal (one partly inside a key tile with queries)
    assert torch.all(dk[:, 200:] == 0) and torch.all(dv[:, 200:] == 0)
    assert torch.all(dk[:, :200].abs().amax(dim=-1) > 0)


def _thd_and_bshd_agree(d, dv, mask, backward):
    import torch

    import scaled_dot_product_02_gb300 as sdpa

    g = _gen(31 * d + dv + len(mask))
    lens = [300, 1, 129, 64]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    t = sum(lens)
    q = _randn(g, t, 4, d)
    k = _randn(g, t, 2, d)
    v = _randn(g, t, 2, dv)
    do = _randn(g, t, 4, dv)
    kw = dict(layout="thd", mask=mask, cu_seqlens_q=cu, cu_seqlens_kv=cu, max_seqlen_q=300, max_seqlen_kv=300)
    o, lse = sdpa.sdpa_fwd(q, k, v, **kw)
    grads = sdpa.sdpa_bwd(q, k, v, o, lse, do, deterministic=True, **kw) if backward else None
    assert sdpa.sdpa_get_device_error() == 0
    for b, (a, e) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        qs, ks, vs, dos = (x[a:e].unsqueeze(0).contiguous() for x in (q, k, v, do))
        ob, lb = sdpa.sdpa_fwd(qs, ks, vs, mask=mask)
        assert torch.equal(ob[0], o[a:e]), f"O of sequence {b}"
        assert torch.equal(lb, lse[a:e]), f"LSE of sequence {b}"
        if backward:
            gb = sdpa.sdpa_bwd(qs, ks, vs, ob, lb, dos, mask=mask, deterministic=True)
            for name, x, y in zip(("dQ", "dK", "dV"), gb, grads):
                assert torch.equal(x[0], y[a:e]), f"{name} of sequence {b}"
    assert sdpa.sdpa_get_device_error() == 0


@pytest.mark.parametrize("d,mask", [(128, "causal"), (128, "causal_br"), (256, "causal"), (512, "none")])
def test_thd_sequences_equal_batch_one_bshd_runs_bit_for_bit(d, mask):
    _thd_and_bshd_agree(d, d, mask, backward=True)


def test_thd_sequences_equal_bshd_runs_asymmetric_forward():
    _thd_and_bshd_agree(192, 128, "causal", backward=False)


@pytest.mark.parametrize("d,deterministic", [(128, False), (128, True), (256, False), (192, None)])
def test_nothing_past_the_output_rows_is_written(d, deterministic):
    import torch

    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_fwd, sdpa_get_device_error

    dv_ = 128 if d == 192 else d
    g = _gen(d + 3)
    lens = [130, 0, 257]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    t, pad = sum(lens), 200
    q = _randn(g, t, 4, d)
    k = _randn(g, t, 2, d)
    v = _randn(g, t, 2, dv_)
    do = _randn(g, t, 4, dv_)
    kw = dict(layout="thd", mask="causal", cu_seqlens_q=cu, cu_seqlens_kv=cu, max_seqlen_q=257, max_seqlen_kv=257)
    canary = 7.0
    o_big = torch.full((t + pad, 4, dv_), canary, dtype=torch.bfloat16, device="cuda")
    l_big = torch.full((t + pad, 4), canary, dtype=torch.float32, device="cuda")
    o, lse = sdpa_fwd(q, k, v, out=o_big[:t], lse=l_big[:t], **kw)
    assert sdpa_get_device_error() == 0
    assert torch.all(o_big[t:] == canary) and torch.all(l_big[t:] == canary)
    assert not torch.any(o_big[:t] == canary)
    if deterministic is None:
        return
    dq_big = torch.full((t + pad, 4, d), canary, dtype=torch.bfloat16, device="cuda")
    dk_big = torch.full((t + pad, 2, d), canary, dtype=torch.bfloat16, device="cuda")
    dv_big = torch.full((t + pad, 2, d), canary, dtype=torch.bfloat16, device="cuda")
    sdpa_bwd(q, k, v, o, lse, do, dq=dq_big[:t], dk=dk_big[:t], dv=dv_big[:t], deterministic=deterministic, **kw)
    assert sdpa_get_device_error() == 0
    for x in (dq_big, dk_big, dv_big):
        assert torch.all(x[t:] == canary)
