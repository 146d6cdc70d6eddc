"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/sdpa.h declares, and declines problems on the host as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module")
def pkg():
    from scaled_dot_product_02_gb300 import build

    build.build()
    import scaled_dot_product_02_gb300 as p

    p.lib()
    return p


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SDPA_API\s+[\w\s\*]+?\b(sdpa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("sdpa_fwd", "sdpa_bwd", "sdpa_fwd_workspace_size", "sdpa_bwd_workspace_size",
                     "sdpa_get_device_error", "sdpa_error_string"):
        assert required in names


def test_library_exports_every_declared_symbol(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(pkg.EXPORTS)


def test_checked_library_exports_every_declared_symbol(pkg):
    """The address-checked build (same sources, SDPA_ADDR_CHECK) is a drop-in
    for libsdpa.so: the same entry points and the same host-side checks."""
    lib = ctypes.CDLL(pkg.CHECKED_LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    with pkg.address_checked():
        assert pkg.lib()._name == pkg.CHECKED_LIB_PATH
        assert pkg.lib().sdpa_check_problem(ctypes.byref(problem(pkg))) == 0
        assert pkg.lib().sdpa_check_problem(ctypes.byref(problem(pkg, head_dim=96))) == 2
        assert pkg.lib().sdpa_debug_address_shrink(-1) == 1  # SDPA_ERR_INVALID_ARG
        assert pkg.lib().sdpa_debug_address_shrink(0) == 0
    assert pkg.lib()._name == pkg.LIB_PATH


def test_normal_library_declines_the_address_checks(pkg):
    assert pkg.lib().sdpa_debug_address_shrink(0) == 2  # SDPA_ERR_UNSUPPORTED
    v = ctypes.c_ulonglong(0)
    assert pkg.lib().sdpa_debug_address_report(ctypes.byref(v), None, None) == 2


def test_error_strings(pkg):
    for code in range(10):
        assert pkg.error_string(code)
    assert pkg.error_string(0) == "ok"
    assert "address" in pkg.error_string(9)


def problem(pkg, **kw):
    p = pkg.Problem()
    base = dict(layout=0, dtype=0, mask_type=1, batch=2, seqlen_q=256, seqlen_kv=256, total_q=0, total_kv=0,
                num_heads_q=8, num_heads_kv=2, head_dim=128, window_left=-1, window_right=-1, softmax_scale=0.088,
                deterministic=0, kv_chunk=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


def test_check_problem_accepts_and_declines(pkg):
    ok = lambda **kw: pkg.sdpa_check_problem(problem(pkg, **kw))
    assert ok() == 0
    assert ok(head_dim=512, mask_type=2, seqlen_q=2048, seqlen_kv=8192) == 0
    assert ok(layout=2, total_q=1000, total_kv=1000) == 0
    assert ok(head_dim=64) == 2                                  # unsupported head dim
    assert ok(head_dim=192) == 2
    assert ok(dtype=5) == 2
    assert ok(num_heads_q=6, num_heads_kv=4) == 1               # Hq % Hkv
    assert ok(window_right=3) == 1                              # causal with a right window
    assert ok(mask_type=0, window_left=16, seqlen_kv=300) == 2  # ambiguous non-causal window alignment
    assert ok(mask_type=0, window_left=16, window_right=16) == 0
    assert ok(window_left=-2) == 1
    assert ok(softmax_scale=float("inf")) == 1
    assert ok(seqlen_kv=0) == 1
    assert ok(layout=7) == 1
    assert ok(deterministic=1) == 0
    assert ok(deterministic=2) == 1
    # head_dim_v: 0 or head_dim is symmetric; (192, 128) is the one asymmetric pair (forward only)
    assert ok(head_dim_v=128) == 0
    assert ok(head_dim=192, head_dim_v=128) == 0
    assert ok(head_dim=192, head_dim_v=128, layout=2, total_q=1000, total_kv=1000) == 0
    assert ok(head_dim=192, head_dim_v=192) == 2
    assert ok(head_dim=128, head_dim_v=192) == 2
    assert ok(head_dim=256, head_dim_v=128) == 2
    assert ok(head_dim_v=-1) == 1


def test_asymmetric_head_dims_are_forward_only(pkg):
    """The backward declines d_qk != d_v before any CUDA call; the forward's
    workspace is the THD guard only (no persistent tile counter)."""
    import ctypes

    L = pkg.lib()
    p = problem(pkg, head_dim=192, head_dim_v=128)
    assert pkg.sdpa_fwd_workspace_size(p) == 0
    assert pkg.sdpa_fwd_workspace_size(problem(pkg, head_dim=192, head_dim_v=128, layout=2, total_q=100,
                                               total_kv=100)) == 256
    assert pkg.sdpa_bwd_workspace_size(p) == 0
    ptr = ctypes.c_void_p
    base = 1 << 40
    args = [ptr(base + i * (1 << 24)) for i in range(9)]
    assert L.sdpa_bwd(ctypes.byref(p), *args, None, None, ptr(base + (1 << 30)), 1 << 20, None) == 2
    assert L.sdpa_bwd_noalloc(ctypes.byref(p), *args, None, None, None) == 2
    # the forward sizes V and O by head_dim_v: an O that would overlap V at D = 192 but not at 128
    p1 = problem(pkg, batch=1, seqlen_q=256, seqlen_kv=256, num_heads_q=2, num_heads_kv=2, head_dim=192,
                 head_dim_v=128)
    nv = 256 * 2 * 128 * 2     # bytes of V [1, 256, 2, 128]
    nq = 256 * 2 * 192 * 2     # bytes of Q or K [1, 256, 2, 192]
    q, k, v = base, base + nq, base + 2 * nq
    o, lse = v + nv, v + nv + nv
    f = lambda o_, lse_: L.sdpa_fwd(ctypes.byref(p1), ptr(q), ptr(k), ptr(v), ptr(o_), ptr(lse_), None, None,
                                    None, 0, None)
    assert f(o - 256, lse) == 4          # o starts inside v
    assert f(o, o + nv - 256) == 4       # lse inside o (o is nv bytes long)


def test_workspace_sizes(pkg):
    p = problem(pkg)
    # head_dim 128 keeps the persistent kernel's tile counter in the workspace
    assert pkg.sdpa_fwd_workspace_size(p) == 256
    assert pkg.sdpa_fwd_workspace_size(problem(pkg, head_dim=256)) == 0
    t = problem(pkg, layout=2, total_q=1000, total_kv=1000)
    assert pkg.sdpa_fwd_workspace_size(t) >= 4
    ws = pkg.sdpa_bwd_workspace_size(p)
    # dQ accumulator (fp32, rows x Hq x D) plus two padded statistics arrays
    assert ws >= 2 * 256 * 8 * 128 * 4 + 2 * 8 * 512 * 4
    assert ws % 256 == 0
    assert pkg.sdpa_bwd_workspace_size(problem(pkg, head_dim=64)) == 0
    # the deterministic head_dim 128 backward writes dQ directly: no fp32 accumulator
    det = pkg.sdpa_bwd_workspace_size(problem(pkg, deterministic=1))
    assert 0 < det < ws and ws - det >= 2 * 256 * 8 * 128 * 4


def test_fp8_workspace_sizes(pkg):
    # guard word and ticket counter (256 bytes), then V transposed to [Hkv][D][keys]: BSHD rounds each
    # sequence's keys up to 16
    for d in (128, 256):
        assert pkg.sdpa_fwd_fp8_workspace_size(problem(pkg, head_dim=d, seqlen_kv=250)) == 256 + 2 * d * 2 * 256
    # THD: every sequence starts on a multiple of 16 (total + 16 per sequence, rounded up)
    t = problem(pkg, head_dim=256, layout=2, total_q=1000, total_kv=1000)
    assert pkg.sdpa_fwd_fp8_workspace_size(t) == 256 + 2 * 256 * 1040
    for d, dv in ((512, 0), (192, 128), (256, 128)):
        assert pkg.sdpa_fwd_fp8_workspace_size(problem(pkg, head_dim=d, head_dim_v=dv)) == 0


def test_kv_chunk_is_validated(pkg):
    for bad in (-128, 1, 100, 129):
        assert pkg.sdpa_check_problem(problem(pkg, head_dim=512, kv_chunk=bad)) == 1
    for good in (0, 128, 1024):
        assert pkg.sdpa_check_problem(problem(pkg, head_dim=512, kv_chunk=good)) == 0


@pytest.mark.parametrize("d,mask", [(512, 2), (512, 0), (256, 1)])
def test_big_backward_workspace_does_not_grow_with_the_keys(pkg, d, mask):
    """head_dim 256/512: the score tiles are held one chunk of keys at a time
    (TransformerEngine PR #3527, "Known limitations": the workspace, not the
    compute, caps the prior art's context length), so past one chunk the
    backward workspace is the same for every key length."""
    base = dict(head_dim=d, mask_type=mask, batch=2, seqlen_q=2048, num_heads_q=16, num_heads_kv=4)
    sizes = [pkg.sdpa_bwd_workspace_size(problem(pkg, seqlen_kv=sk, **base)) for sk in (8192, 16384, 65536, 262144)]
    assert len(set(sizes)) == 1 and sizes[0] > 0, sizes
    assert sizes[0] < (1 << 30)  # the 8192-key D512 workload would hold 4 GiB of tiles unchunked
    # a short key range fits one chunk and needs less
    assert pkg.sdpa_bwd_workspace_size(problem(pkg, seqlen_kv=512, **base)) < sizes[0]
    # a caller-chosen chunk bounds it further; chunking adds the fp32 dQ accumulator
    small = pkg.sdpa_bwd_workspace_size(problem(pkg, seqlen_kv=65536, kv_chunk=128, **base))
    tile_pairs = 2 * 16 * 16  # (batch, q head, q tile) x one key tile
    acc = 2 * 2048 * 16 * d * 4
    assert small < sizes[0] and small >= acc + tile_pairs * 65536  # a 16-bit P and dS image per pair


def test_window_bounds_the_big_backward_workspace(pkg):
    """A bounded window already bounds the keys a query tile sees: the tile
    arrays hold the window's span, whatever the key length."""
    base = dict(head_dim=256, mask_type=1, batch=2, num_heads_q=16, num_heads_kv=8, window_left=1024, window_right=0)
    sizes = {sk: pkg.sdpa_bwd_workspace_size(problem(pkg, seqlen_q=sk, seqlen_kv=sk, **base)) for sk in (8192, 16384)}
    per_q_tile = (sizes[16384] - sizes[8192]) / ((16384 - 8192) // 128)
    # per added query tile: 11 slots of P and dS for every (batch, head), plus statistics
    assert abs(per_q_tile - 2 * 16 * 11 * 65536) < 2 * 16 * 128 * 8 + 4096


def test_product_path_refuses_cpu_tensors(pkg):
    import torch

    q = torch.zeros(1, 128, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkg.sdpa_fwd(q, q, q, mask="causal")


def test_host_validation_before_any_cuda_call(pkg):
    """Alignment, null-pointer, workspace and overlap checks return before the
    library touches CUDA, so they run here with made-up addresses."""
    import ctypes

    L = pkg.lib()
    p = problem(pkg, batch=1, seqlen_q=256, seqlen_kv=256, num_heads_q=2, num_heads_kv=2)
    n = 256 * 2 * 128 * 2  # bytes of one 16-bit [1, 256, 2, 128] tensor
    base = 1 << 40
    q, k, v, o = base, base + n, base + 2 * n, base + 3 * n
    lse = base + 4 * n
    ptr = ctypes.c_void_p
    wsf = base + (1 << 31)
    call = lambda *a: L.sdpa_fwd(ctypes.byref(p), *[ptr(x) if x is not None else None for x in a], 256, None)
    assert call(q + 8, k, v, o, lse, None, None, wsf) == 3         # misaligned q
    assert call(q, k, v, o, lse + 4, None, None, wsf) == 3         # misaligned lse
    assert call(None, k, v, o, lse, None, None, wsf) == 1          # null input
    assert call(q, k, v, q + 64, lse, None, None, wsf) == 4        # o overlaps q
    assert call(q, k, v, o, o + 16, None, None, wsf) == 4          # lse overlaps o
    assert call(q, k, v, o, lse, None, None, None) == 5            # head_dim 128 needs its workspace
    t = problem(pkg, layout=2, batch=2, seqlen_q=128, seqlen_kv=128, total_q=256, total_kv=256, num_heads_q=2,
                num_heads_kv=2)
    ws = pkg.sdpa_fwd_workspace_size(t)
    assert ws > 0
    rc = L.sdpa_fwd(ctypes.byref(t), ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(base + 8 * n), ptr(base + 9 * n),
                    None, 0, None)
    assert rc == 5                                                 # THD needs its guard workspace
    rc = L.sdpa_fwd(ctypes.byref(t), ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), None, None, ptr(base + 10 * n), ws,
                    None)
    assert rc == 1                                                 # THD without cu_seqlens
    # backward: workspace too small, and an output overlapping the workspace
    wsb = pkg.sdpa_bwd_workspace_size(p)
    bcall = lambda wsp, wsz, dq: L.sdpa_bwd(ctypes.byref(p), ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(o),
                                            ptr(dq), ptr(base + 7 * n), ptr(base + 8 * n), None, None, ptr(wsp), wsz,
                                            None)
    ws0 = base + (1 << 30)
    assert bcall(ws0, wsb - 256, base + 6 * n) == 5
    assert bcall(ws0, wsb, ws0 + 256) == 4
    assert bcall(ws0 + 16, wsb, base + 6 * n) == 3                 # workspace must be 256-byte aligned


def test_zero_sized_problems_are_no_ops(pkg):
    import ctypes

    p = problem(pkg, batch=0)
    assert pkg.lib().sdpa_fwd(ctypes.byref(p), None, None, None, None, None, None, None, None, 0, None) == 0


def test_merge_host_validation(pkg):
    """sdpa_merge declines on the host before any CUDA call."""
    import ctypes

    L = pkg.lib()
    ptr = ctypes.c_void_p
    base = 1 << 40
    items, d = 1000, 128
    ob, lb = items * d * 2, items * 4
    po, pl, o, lse = base, base + 4 * ob, base + 8 * ob, base + 9 * ob

    def call(n_parts=3, dtype=0, head_dim=d, n_items=items, a=po, b=pl, c=o, e=lse):
        p = pkg.MergeProblem(dtype, n_items, head_dim, n_parts)
        return L.sdpa_merge(ctypes.byref(p), ptr(a), ptr(b), ptr(c), ptr(e), None)

    assert call(n_parts=0) == 1                      # SDPA_ERR_INVALID_ARG
    assert call(n_parts=65) == 1
    assert call(head_dim=64) == 2                    # SDPA_ERR_UNSUPPORTED
    assert call(dtype=3) == 2
    assert call(n_items=0) == 0                      # nothing to do
    assert call(a=po + 8) == 3                       # SDPA_ERR_ALIGNMENT
    assert call(c=po + ob) == 4                      # output inside the partial outputs: SDPA_ERR_OVERLAP
    assert call(e=pl) == 4                           # output LSE over the partial LSE
    assert L.sdpa_merge(None, None, None, None, None, None) == 1


def test_binding_refuses_inconsistent_tensors_before_any_device_access(pkg):
    """The binding checks shapes, dtypes and devices from tensor metadata, so
    a tensor smaller than the problem it belongs to never reaches a kernel."""
    import torch

    bf = torch.bfloat16
    q = torch.zeros(2, 64, 4, 128, dtype=bf)
    k = torch.zeros(2, 96, 2, 128, dtype=bf)
    v = torch.zeros(2, 96, 2, 128, dtype=bf)
    ok = lambda **kw: pkg._validate("bshd", q, k, v, **kw)
    ok()
    ok(o=torch.zeros(2, 64, 4, 128, dtype=bf), lse=torch.zeros(128, 4), dout=torch.zeros(2, 64, 4, 128, dtype=bf),
       dq=torch.zeros_like(q), dk=torch.zeros_like(k), dv=torch.zeros_like(v))
    pkg._validate("bshd", torch.zeros(1, 8, 2, 192, dtype=bf), torch.zeros(1, 8, 2, 192, dtype=bf),
                  torch.zeros(1, 8, 2, 128, dtype=bf), o=torch.zeros(1, 8, 2, 128, dtype=bf))  # 192/128
    bad = [
        lambda: pkg._validate("bshd", q, k, torch.zeros(2, 95, 2, 128, dtype=bf)),               # v shorter than k
        lambda: pkg._validate("bshd", q, torch.zeros(2, 96, 2, 64, dtype=bf), v),                # head_dim mismatch
        lambda: pkg._validate("bshd", q, torch.zeros(1, 96, 2, 128, dtype=bf),
                              torch.zeros(1, 96, 2, 128, dtype=bf)),                             # batch mismatch
        lambda: pkg._validate("bshd", q, k.half(), v),                                           # dtype mismatch
        lambda: pkg._validate("bshd", q.float(), k.float(), v.float()),                          # fp32 inputs
        lambda: pkg._validate("thd", q, k, v),                                                   # rank for thd
        lambda: ok(o=torch.zeros(2, 64, 4, 64, dtype=bf)),                                       # o too narrow
        lambda: ok(lse=torch.zeros(128, 4, dtype=torch.float64)),                                # lse dtype
        lambda: ok(lse=torch.zeros(127, 4)),                                                     # lse rows
        lambda: ok(dout=torch.zeros(2, 63, 4, 128, dtype=bf)),                                   # dO shape
        lambda: ok(dk=torch.zeros(2, 96, 2, 128, dtype=torch.float16)),                          # dK dtype
        lambda: pkg._validate("thd", q[0], k[0], v[0], cu_q=torch.zeros(3, dtype=torch.int64)),  # cu dtype
        lambda: pkg._validate("thd", q[0], k[0], v[0], cu_q=torch.zeros(3, dtype=torch.int32),
                              cu_kv=torch.zeros(4, dtype=torch.int32)),                          # cu lengths
    ]
    for i, f in enumerate(bad):
        with pytest.raises(ValueError):
            f()
    # merge: an output smaller than one block's rows is refused too
    po = torch.zeros(3, 10, 2, 128, dtype=bf)
    pl = torch.zeros(3, 10, 2)
    with pytest.raises(ValueError):
        pkg.sdpa_merge(po, pl, out=torch.zeros(9, 2, 128, dtype=bf))
    with pytest.raises(ValueError):
        pkg.sdpa_merge(po, pl, out=torch.zeros(10, 2, 128, dtype=torch.float16))


def test_missing_library_fails_loudly_with_no_fallback(tmp_path):
    """In a fresh interpreter whose package copy has no libsdpa.so, every entry
    point raises ImportError: there is no other implementation to fall back to."""
    import shutil
    import subprocess
    import sys

    pkg_src = os.path.join(ROOT, "scaled_dot_product_02_gb300", "__init__.py")
    dst = tmp_path / "scaled_dot_product_02_gb300"
    dst.mkdir()
    shutil.copy(pkg_src, dst / "__init__.py")
    code = ("import scaled_dot_product_02_gb300 as s, torch\n"
            "q = torch.zeros(1, 128, 2, 128, dtype=torch.bfloat16)\n"
            "for f in (lambda: s.lib(), lambda: s.sdpa_fwd(q, q, q)):\n"
            "    try:\n"
            "        f()\n"
            "    except ImportError as e:\n"
            "        print('raised', 'libsdpa.so' in str(e))\n"
            "    else:\n"
            "        print('no error')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split("\n")[:2] == ["raised True", "raised True"], r.stdout


def _header_struct(name, path=HEADER):
    """(field, C type) pairs of `typedef struct { ... } name;` in a C source, in order."""
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    body = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + r"\s*;", text).group(1)
    fields = []
    for decl in body.split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        m = re.match(r"((?:unsigned |long |short )*\w+)\s+(.*)", decl)
        ctype, names = m.group(1), m.group(2)
        fields += [(n.strip(), ctype) for n in names.split(",")]
    return fields


def test_ctypes_structs_mirror_the_header(pkg):
    """The binding's ctypes structures must match the C structs field for
    field (name, order and type), or every call would pass shifted values."""
    import ctypes

    ctype_of = {"int": ctypes.c_int, "float": ctypes.c_float, "long long": ctypes.c_longlong}
    for cname, py in (("sdpa_problem", pkg.Problem), ("sdpa_merge_problem", pkg.MergeProblem)):
        want = _header_struct(cname)
        got = [(f, t) for f, t in py._fields_]
        assert [f for f, _ in got] == [f for f, _ in want], cname
        for (f, t), (_, ct) in zip(got, want):
            assert t is ctype_of[ct], (cname, f, ct)


def test_oracle_ctypes_struct_mirrors_its_c_struct():
    import ctypes

    from oracle import oracle

    ctype_of = {"int": ctypes.c_int, "double": ctypes.c_double}
    want = _header_struct("oracle_problem", os.path.join(ROOT, "oracle", "sdpa_oracle.c"))
    got = list(oracle._Problem._fields_)
    assert [f for f, _ in got] == [f for f, _ in want]
    for (f, t), (_, ct) in zip(got, want):
        assert t is ctype_of[ct], (f, ct)


def test_a_plain_c_program_uses_the_abi(pkg, tmp_path):
    """tests/c_abi_host_check.c, compiled as C99 by gcc against include/sdpa.h
    and linked to libsdpa.so, runs its host-side checks (no GPU needed)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / "c_abi_host_check")
    libdir = os.path.dirname(pkg.LIB_PATH)
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c_abi_host_check.c"), "-o", exe, "-L", libdir, "-lsdpa",
                           f"-Wl,-rpath,{libdir}"])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
