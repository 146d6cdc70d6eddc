"""Out-of-bounds stand-in: the address-checked library.

compute-sanitizer's memory checker is closed on this machine, and element-wise
parity cannot see a store that lands outside every output (PR #3705, "sync
qualification", records a bug that numerics passed and only a sanitizer
caught). libsdpa_checked.so is the same sources compiled with SDPA_ADDR_CHECK:
each entry point registers the byte extents of the buffers it was given, and
every kernel load or store at a computed global address first tests its bytes
against them, skipping and recording any access outside (tensor-map copies are
bounded by the hardware against their maps).

  * Every entry point on representative cases (D128/256/512, BSHD/SBHD/THD,
    GQA, masks, windows, key chunks, deterministic, no-alloc, FP8, merge,
    the 192/128 forward) runs through the checked library with no violation,
    and gives the same bits as the normal library.
  * With every registered extent pulled in by 16 bytes (the memory itself
    stays valid), the forward's last stores are rejected, counted and
    skipped: the checker sees accesses and nothing is written past the
    shortened extents.
"""
import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("d128_thd_gqa", "thd", "causal", 4, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300)), {}),
    (Workload("d128_sbhd_fp16_nomask", "sbhd", "none", 2, 200, 200, 2, 2, 128, "fp16", std=0.5), {}),
    (Workload("d128_bshd_br_deterministic", "bshd", "causal_br", 1, 200, 333, 4, 1, 128, "bf16"),
     {"deterministic": True}),
    (Workload("d256_window", "bshd", "causal", 1, 400, 400, 2, 1, 256, "bf16", window=(100, 0)), {}),
    (Workload("d512_thd_chunks", "thd", "causal", 3, 300, 300, 2, 1, 512, "bf16", len_range=(1, 300)),
     {"kv_chunk": 128}),
]


def _fwd_bwd(w, inp, bwd_kw, noalloc=False):
    from parity import gpu_kwargs, to_device
    from scaled_dot_product_02_gb300 import sdpa_bwd, sdpa_bwd_noalloc, sdpa_fwd, sdpa_get_device_error

    q, k, v, do = (to_device(inp[x], w.dtype) for x in ("q", "k", "v", "do"))
    kw = gpu_kwargs(w, inp)
    o, lse = sdpa_fwd(q, k, v, **kw)
    bwd = sdpa_bwd_noalloc if noalloc else sdpa_bwd
    grads = bwd(q, k, v, o, lse, do, **bwd_kw, **kw)
    assert sdpa_get_device_error() == 0
    return (o, lse) + tuple(grads)


def _no_violations():
    import scaled_dot_product_02_gb300 as sdpa

    n, addr, size = sdpa.sdpa_debug_address_report()
    assert n == 0, f"{n} accesses outside the call's buffers, first at {addr:#x} ({size} bytes)"
    assert sdpa.sdpa_get_device_error() == 0


def _same(a, b):
    import torch

    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x, y), f"output {i} differs between the normal and the checked library"


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_checked_library_sees_no_stray_access(case):
    import scaled_dot_product_02_gb300 as sdpa

    w, bwd_kw = case
    inp = workloads.make_inputs(w, seed=83)
    ref = _fwd_bwd(w, inp, bwd_kw)
    with sdpa.address_checked():
        sdpa.sdpa_debug_address_report()  # start from a clean count
        got = _fwd_bwd(w, inp, bwd_kw)
        _no_violations()
    exact = [True, True, w.head_dim != 128 or bwd_kw.get("deterministic", False), True, True]
    import torch

    for i, (x, y, ex) in enumerate(zip(got, ref, exact)):
        if ex:
            assert torch.equal(x, y), f"output {i} differs between the normal and the checked library"
        else:  # dQ of the D128 backward: fp32 reductions in arrival order
            diff = (x.float() - y.float()).abs().max().item()
            assert diff <= 2.0 ** -8 * max(1.0, y.float().abs().max().item()), diff


def test_checked_library_other_entry_points():
    import torch

    import scaled_dot_product_02_gb300 as sdpa
    from parity import gpu_kwargs, to_device

    # allocation-free backward (its scratch is a static array of the library)
    w = Workload("noalloc_thd", "thd", "causal", 3, 200, 200, 4, 2, 128, "bf16", len_range=(1, 200))
    inp = workloads.make_inputs(w, seed=85)
    ref = _fwd_bwd(w, inp, {}, noalloc=True)
    # FP8 forward, head_dim 128 and 256
    wf = Workload("fp8_thd", "thd", "causal", 3, 300, 300, 4, 2, 128, "bf16", len_range=(1, 300))
    f8 = workloads.fp8_inputs(wf, seed=87)
    q8, k8, v8 = (torch.from_numpy(f8[x]).cuda() for x in ("q8", "k8", "v8"))
    ref8 = sdpa.sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, **gpu_kwargs(wf, f8))
    wf2 = Workload("fp8_d256_bshd", "bshd", "causal", 2, 300, 300, 4, 2, 256, "bf16")
    f82 = workloads.fp8_inputs(wf2, seed=88)
    q82, k82, v82 = (torch.from_numpy(f82[x]).cuda() for x in ("q8", "k8", "v8"))
    ref82 = sdpa.sdpa_fwd_fp8(q82, k82, v82, descale=workloads.FP8_DESCALE, **gpu_kwargs(wf2, f82))
    # 192/128 forward
    wa = Workload("asym", "thd", "causal", 3, 200, 200, 4, 2, 192, "bf16", len_range=(1, 200), head_dim_v=128)
    ia = workloads.make_inputs(wa, seed=89)
    qa, ka, va = (to_device(ia[x], wa.dtype) for x in ("q", "k", "v"))
    refa = sdpa.sdpa_fwd(qa, ka, va, **gpu_kwargs(wa, ia))
    # merge of two key halves
    parts = torch.randn(2, 300, 4, 128, device="cuda").to(torch.bfloat16)
    lses = torch.randn(2, 300, 4, device="cuda")
    lses[0, :7] = -float("inf")
    refm = sdpa.sdpa_merge(parts, lses)
    with sdpa.address_checked():
        sdpa.sdpa_debug_address_report()
        got = _fwd_bwd(w, inp, {}, noalloc=True)
        _no_violations()
        got8 = sdpa.sdpa_fwd_fp8(q8, k8, v8, descale=workloads.FP8_DESCALE, **gpu_kwargs(wf, f8))
        _no_violations()
        got82 = sdpa.sdpa_fwd_fp8(q82, k82, v82, descale=workloads.FP8_DESCALE, **gpu_kwargs(wf2, f82))
        _no_violations()
        gota = sdpa.sdpa_fwd(qa, ka, va, **gpu_kwargs(wa, ia))
        _no_violations()
        gotm = sdpa.sdpa_merge(parts, lses)
        _no_violations()
    _same(got[:2] + got[3:], ref[:2] + ref[3:])
    _same(got8, ref8)
    _same(got82, ref82)
    _same(gota, refa)
    _same(gotm, refm)


def test_checker_rejects_and_skips_accesses_outside_the_extents():
    import torch

    import scaled_dot_product_02_gb300 as sdpa
    from parity import gpu_kwargs, to_device

    w = Workload("shrunk", "bshd", "causal", 1, 256, 256, 2, 2, 128, "bf16")
    inp = workloads.make_inputs(w, seed=91)
    q, k, v = (to_device(inp[x], w.dtype) for x in ("q", "k", "v"))
    o_ref, lse_ref = sdpa.sdpa_fwd(q, k, v, **gpu_kwargs(w, inp))
    o = torch.full_like(o_ref, 7.0)
    lse = torch.full_like(lse_ref, 7.0)
    with sdpa.address_checked():
        sdpa.sdpa_debug_address_report()
        try:
            sdpa.sdpa_debug_address_shrink(16)
            sdpa.sdpa_fwd(q, k, v, out=o, lse=lse, **gpu_kwargs(w, inp))
            n, addr, size = sdpa.sdpa_debug_address_report()
            err = sdpa.sdpa_get_device_error()
        finally:
            sdpa.sdpa_debug_address_shrink(0)
        assert err == 9, err  # SDPA_ERR_ADDRESS
        assert n > 0
        o_end = o.data_ptr() + o.numel() * o.element_size()
        l_end = lse.data_ptr() + lse.numel() * lse.element_size()
        assert o_end - 64 <= addr < o_end or l_end - 16 <= addr < l_end, (hex(addr), size)
        # the last 16 bytes of both outputs were never written; the rest was
        ob = o.view(torch.uint8).flatten()
        rb = o_ref.view(torch.uint8).flatten()
        sentinel = torch.full_like(o_ref, 7.0).view(torch.uint8).flatten()
        assert torch.equal(ob[-16:], sentinel[-16:])
        assert torch.equal(ob[:-64], rb[:-64])
        lf, lr = lse.flatten(), lse_ref.flatten()
        assert torch.all(lf[-4:] == 7.0) and torch.equal(lf[:-4], lr[:-4])
        # unshrunk again: a clean run
        sdpa.sdpa_fwd(q, k, v, out=o, lse=lse, **gpu_kwargs(w, inp))
        _no_violations()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
