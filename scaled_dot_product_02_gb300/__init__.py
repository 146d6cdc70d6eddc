"""Python binding of libsdpa.so, the fused SDPA library for one GB300 GPU.

The functions carry the C ABI's names (include/sdpa.h) and only marshal
arguments: torch supplies device memory and the current CUDA stream, and every
step of the computation runs in the library's CUDA kernels. There is no other
implementation behind these calls: if libsdpa.so is missing, or the tensors
are not CUDA tensors, the call raises.

Layouts: "bshd" [B,S,H,D], "sbhd" [S,B,H,D], "thd" [T,H,D] (+ cu_seqlens).
Masks: "none", "causal" (top-left), "causal_br" (bottom-right).
V (and O, dO) may be narrower than Q/K for the forward's 192/128 pair; the
binding reads that width from v. Tensor shapes, dtypes and devices are checked
against each other from metadata before the library is called.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsdpa.so")
CHECKED_LIB_PATH = os.path.join(PKG, "libsdpa_checked.so")  # the address-checked testing build

LAYOUTS = {"bshd": 0, "sbhd": 1, "thd": 2}
MASKS = {"none": 0, "causal": 1, "causal_br": 2}
STATUS = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARG", 2: "SDPA_ERR_UNSUPPORTED", 3: "SDPA_ERR_ALIGNMENT",
          4: "SDPA_ERR_OVERLAP", 5: "SDPA_ERR_WORKSPACE_TOO_SMALL", 6: "SDPA_ERR_BAD_SEQLENS",
          7: "SDPA_ERR_TIMEOUT", 8: "SDPA_ERR_CUDA", 9: "SDPA_ERR_ADDRESS"}
EXPORTS = ("sdpa_fwd_workspace_size", "sdpa_bwd_workspace_size", "sdpa_check_problem", "sdpa_fwd", "sdpa_bwd",
           "sdpa_get_device_error", "sdpa_error_string", "sdpa_last_launch_count", "sdpa_profile_begin",
           "sdpa_profile_end", "sdpa_bwd_noalloc", "sdpa_selftest_bounded_wait", "sdpa_merge",
           "sdpa_fwd_fp8_workspace_size", "sdpa_fwd_fp8", "sdpa_debug_set_max_ctas", "sdpa_debug_address_report",
           "sdpa_debug_address_shrink")
NOALLOC_MAX_BYTES = 32 << 20  # SDPA_BWD_NOALLOC_MAX_BYTES
KERNEL_KINDS = ("fwd", "bwd", "preprocess", "dq_finalize", "guard", "merge", "bwd_dq", "v_transpose")


class SdpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({error_string(status)})")


class MergeProblem(ctypes.Structure):
    """sdpa_merge_problem (include/sdpa.h)."""
    _fields_ = [("dtype", ctypes.c_int), ("items", ctypes.c_longlong), ("head_dim", ctypes.c_int),
                ("n_parts", ctypes.c_int)]


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("layout", "dtype", "mask_type", "batch", "seqlen_q", "seqlen_kv",
                                            "total_q", "total_kv", "num_heads_q", "num_heads_kv", "head_dim",
                                            "window_left", "window_right")] + [("softmax_scale", ctypes.c_float),
                                                                               ("deterministic", ctypes.c_int),
                                                                               ("head_dim_v", ctypes.c_int),
                                                                               ("kv_chunk", ctypes.c_int)]


_lock = threading.Lock()
_libs = {}
_active = LIB_PATH


def _load(path):
    if path not in _libs:
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: run scaled_dot_product_02_gb300/build.py "
                              "(there is no fallback implementation)")
        L = ctypes.CDLL(path)
        vp, pp = ctypes.c_void_p, ctypes.POINTER(Problem)
        L.sdpa_fwd_workspace_size.argtypes = [pp]
        L.sdpa_fwd_workspace_size.restype = ctypes.c_size_t
        L.sdpa_bwd_workspace_size.argtypes = [pp]
        L.sdpa_bwd_workspace_size.restype = ctypes.c_size_t
        L.sdpa_check_problem.argtypes = [pp]
        L.sdpa_fwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.sdpa_bwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.sdpa_get_device_error.argtypes = [vp]
        L.sdpa_error_string.argtypes = [ctypes.c_int]
        L.sdpa_error_string.restype = ctypes.c_char_p
        L.sdpa_last_launch_count.restype = ctypes.c_int
        L.sdpa_selftest_bounded_wait.argtypes = [ctypes.c_uint, vp]
        L.sdpa_debug_set_max_ctas.argtypes = [ctypes.c_int]
        u64p = ctypes.POINTER(ctypes.c_ulonglong)
        L.sdpa_debug_address_report.argtypes = [u64p, u64p, u64p]
        L.sdpa_debug_address_shrink.argtypes = [ctypes.c_longlong]
        L.sdpa_bwd_noalloc.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sdpa_merge.argtypes = [ctypes.POINTER(MergeProblem), vp, vp, vp, vp, vp]
        L.sdpa_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                                       ctypes.c_int]
        L.sdpa_fwd_fp8_workspace_size.argtypes = [pp]
        L.sdpa_fwd_fp8_workspace_size.restype = ctypes.c_size_t
        fl = ctypes.c_float
        L.sdpa_fwd_fp8.argtypes = [pp, vp, vp, vp, fl, fl, fl, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        _libs[path] = L
    return _libs[path]


def lib():
    """The loaded library every call goes through: libsdpa.so, or
    libsdpa_checked.so inside `address_checked()` (build them first with
    scaled_dot_product_02_gb300.build)."""
    with _lock:
        return _load(_active)


@contextlib.contextmanager
def address_checked():
    """Testing aid: route the calls made inside the block through
    libsdpa_checked.so, whose kernels test every computed global access
    against the call's buffers (sdpa_debug_address_report in include/sdpa.h).
    Both libraries stay loaded; each keeps its own device error word."""
    global _active
    with _lock:
        prev, _active = _active, CHECKED_LIB_PATH
        _load(CHECKED_LIB_PATH)
    try:
        yield
    finally:
        with _lock:
            _active = prev


def sdpa_debug_address_report():
    """(violations, first address, its size) since the last report, then
    cleared (synchronises the device). Address-checked library only."""
    v, a, n = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    rc = lib().sdpa_debug_address_report(ctypes.byref(v), ctypes.byref(a), ctypes.byref(n))
    if rc:
        raise SdpaError(rc, "sdpa_debug_address_report")
    return v.value, a.value, n.value


def sdpa_debug_address_shrink(nbytes: int) -> None:
    """Pull the end of every extent registered from now on in by nbytes (0
    restores them). Address-checked library only."""
    rc = lib().sdpa_debug_address_shrink(int(nbytes))
    if rc:
        raise SdpaError(rc, "sdpa_debug_address_shrink")


def error_string(status: int) -> str:
    return lib().sdpa_error_string(int(status)).decode()


sdpa_error_string = error_string


def make_problem(q, k, *, layout="bshd", mask="none", window=(-1, -1), scale=None, dtype=None, batch=None,
                 max_seqlen_q=None, max_seqlen_kv=None, deterministic=False, head_dim_v=0, kv_chunk=0) -> Problem:
    """sdpa_problem from tensor shapes (no device access). head_dim_v: the
    width of V and O rows (0 = Q/K's head_dim). kv_chunk: key positions per
    chunk of the head_dim 256/512 backward (a multiple of 128; 0 = the
    library's choice)."""
    import torch

    if dtype is None:
        dtype = {torch.bfloat16: 0, torch.float16: 1}.get(q.dtype, -1)
    d = q.shape[-1]
    p = Problem()
    p.layout, p.dtype, p.mask_type = LAYOUTS[layout], dtype, MASKS[mask]
    if layout == "bshd":
        p.batch, p.seqlen_q, p.num_heads_q = q.shape[0], q.shape[1], q.shape[2]
        p.seqlen_kv, p.num_heads_kv = k.shape[1], k.shape[2]
    elif layout == "sbhd":
        p.seqlen_q, p.batch, p.num_heads_q = q.shape[0], q.shape[1], q.shape[2]
        p.seqlen_kv, p.num_heads_kv = k.shape[0], k.shape[2]
    else:
        if batch is None or max_seqlen_q is None or max_seqlen_kv is None:
            raise ValueError("thd needs batch, max_seqlen_q and max_seqlen_kv")
        p.batch, p.seqlen_q, p.seqlen_kv = batch, max_seqlen_q, max_seqlen_kv
        p.total_q, p.total_kv = q.shape[0], k.shape[0]
        p.num_heads_q, p.num_heads_kv = q.shape[1], k.shape[1]
    p.head_dim = d
    p.window_left, p.window_right = int(window[0]), int(window[1])
    p.softmax_scale = float(scale if scale is not None else d ** -0.5)
    p.deterministic = int(bool(deterministic))
    p.head_dim_v = int(head_dim_v)
    p.kv_chunk = int(kv_chunk)
    return p


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("sdpa tensors must be CUDA tensors (there is no CPU implementation)")
        if t is not None and not t.is_contiguous():
            raise ValueError("sdpa tensors must be contiguous in their layout")


def _validate(layout, q, k, v, *, o=None, lse=None, dout=None, dq=None, dk=None, dv=None, cu_q=None, cu_kv=None):
    """Shapes, dtypes and devices of one call's tensors, from their metadata
    alone (no device access, no synchronisation). The C ABI receives bare
    pointers and sizes taken from q and k, so a tensor smaller than the
    problem it is part of would let the kernels read or write past its end:
    such calls are refused here with ValueError."""
    import torch

    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"q must be bfloat16 or float16, got {q.dtype}")
    rank = 3 if layout == "thd" else 4
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != rank:
            raise ValueError(f"{name} must have {rank} dimensions in layout {layout}, got {tuple(t.shape)}")
        if t.dtype != q.dtype or t.device != q.device:
            raise ValueError(f"{name} must have q's dtype and device ({q.dtype}, {q.device})")
    if k.shape[-1] != q.shape[-1]:
        raise ValueError(f"q and k must share head_dim, got {q.shape[-1]} and {k.shape[-1]}")
    if tuple(k.shape[:-1]) != tuple(v.shape[:-1]):
        raise ValueError(f"k and v must agree on every dimension but the last, got {tuple(k.shape)} and "
                         f"{tuple(v.shape)}")
    batch_dim = {"bshd": 0, "sbhd": 1}.get(layout)
    if batch_dim is not None and q.shape[batch_dim] != k.shape[batch_dim]:
        raise ValueError(f"q and k must have the same batch size, got {q.shape[batch_dim]} and {k.shape[batch_dim]}")
    o_shape = tuple(q.shape[:-1]) + (v.shape[-1],)
    rows_q = q.numel() // max(1, q.shape[-1] * q.shape[-2])
    for name, t, shape, dtype in (("o", o, o_shape, q.dtype), ("dout", dout, o_shape, q.dtype),
                                  ("dq", dq, tuple(q.shape), q.dtype), ("dk", dk, tuple(k.shape), q.dtype),
                                  ("dv", dv, tuple(v.shape), q.dtype),
                                  ("lse", lse, (rows_q, q.shape[-2]), torch.float32)):
        if t is None:
            continue
        if tuple(t.shape) != shape or t.dtype != dtype or t.device != q.device:
            raise ValueError(f"{name} must be {dtype} of shape {shape} on {q.device}, got {t.dtype} "
                             f"{tuple(t.shape)} on {t.device}")
    for name, t in (("cu_seqlens_q", cu_q), ("cu_seqlens_kv", cu_kv)):
        if t is None:
            continue
        if t.dtype != torch.int32 or t.dim() != 1 or t.numel() < 1 or t.device != q.device:
            raise ValueError(f"{name} must be a 1-D int32 tensor of batch + 1 entries on {q.device}")
    if cu_q is not None and cu_kv is not None and cu_q.numel() != cu_kv.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_kv must have the same number of entries")


def sdpa_check_problem(p: Problem) -> int:
    return int(lib().sdpa_check_problem(ctypes.byref(p)))


def sdpa_fwd_workspace_size(p: Problem) -> int:
    return int(lib().sdpa_fwd_workspace_size(ctypes.byref(p)))


def sdpa_bwd_workspace_size(p: Problem) -> int:
    return int(lib().sdpa_bwd_workspace_size(ctypes.byref(p)))


def sdpa_fwd(q, k, v, *, layout="bshd", mask="none", window=(-1, -1), scale=None, cu_seqlens_q=None,
             cu_seqlens_kv=None, max_seqlen_q=None, max_seqlen_kv=None, out=None, lse=None, workspace=None,
             stream=None):
    """Forward. Returns (o, lse); o has Q's shape with V's last dimension,
    lse is float32 [rows_q, Hq] token-major."""
    import torch

    batch = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_problem(q, k, layout=layout, mask=mask, window=window, scale=scale, batch=batch,
                     max_seqlen_q=max_seqlen_q, max_seqlen_kv=max_seqlen_kv, head_dim_v=v.shape[-1])
    rows_q = q.numel() // (q.shape[-1] * q.shape[-2])
    if out is None:
        out = torch.empty(tuple(q.shape[:-1]) + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((rows_q, q.shape[-2]), dtype=torch.float32, device=q.device)
    _validate(layout, q, k, v, o=out, lse=lse, cu_q=cu_seqlens_q, cu_kv=cu_seqlens_kv)
    need = sdpa_fwd_workspace_size(p)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check_cuda(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sdpa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                        _ptr(cu_seqlens_kv), _ptr(workspace), ws_bytes, _stream(stream))
    if rc:
        raise SdpaError(rc, "sdpa_fwd")
    return out, lse


def sdpa_bwd(q, k, v, o, lse, dout, *, layout="bshd", mask="none", window=(-1, -1), scale=None,
             cu_seqlens_q=None, cu_seqlens_kv=None, max_seqlen_q=None, max_seqlen_kv=None, dq=None, dk=None,
             dv=None, workspace=None, stream=None, deterministic=False, kv_chunk=0):
    """Backward. Returns (dq, dk, dv). deterministic=True makes every
    gradient bitwise reproducible run to run (see sdpa_problem.deterministic);
    kv_chunk sets sdpa_problem.kv_chunk (head_dim 256/512)."""
    import torch

    batch = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_problem(q, k, layout=layout, mask=mask, window=window, scale=scale, batch=batch,
                     max_seqlen_q=max_seqlen_q, max_seqlen_kv=max_seqlen_kv, deterministic=deterministic,
                     head_dim_v=v.shape[-1], kv_chunk=kv_chunk)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _validate(layout, q, k, v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv, cu_q=cu_seqlens_q, cu_kv=cu_seqlens_kv)
    need = sdpa_bwd_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check_cuda(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().sdpa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                        _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(workspace), ws_bytes,
                        _stream(stream))
    if rc:
        raise SdpaError(rc, "sdpa_bwd")
    return dq, dk, dv


def sdpa_bwd_noalloc(q, k, v, o, lse, dout, *, layout="bshd", mask="none", window=(-1, -1), scale=None,
                     cu_seqlens_q=None, cu_seqlens_kv=None, max_seqlen_q=None, max_seqlen_kv=None, dq=None,
                     dk=None, dv=None, stream=None, deterministic=False, kv_chunk=0):
    """Backward without a workspace: the library's static scratch array is
    used instead (for callers that cannot allocate device memory; problems
    needing more than NOALLOC_MAX_BYTES of scratch are rejected). Calls that
    overlap on the GPU race on that array. Returns (dq, dk, dv); pass dq/dk/dv
    to avoid torch allocating them here."""
    import torch

    batch = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_problem(q, k, layout=layout, mask=mask, window=window, scale=scale, batch=batch,
                     max_seqlen_q=max_seqlen_q, max_seqlen_kv=max_seqlen_kv, deterministic=deterministic,
                     head_dim_v=v.shape[-1], kv_chunk=kv_chunk)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _validate(layout, q, k, v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv, cu_q=cu_seqlens_q, cu_kv=cu_seqlens_kv)
    _check_cuda(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv)
    rc = lib().sdpa_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
                                _stream(stream))
    if rc:
        raise SdpaError(rc, "sdpa_bwd_noalloc")
    return dq, dk, dv


def sdpa_fwd_fp8_workspace_size(p: Problem) -> int:
    return int(lib().sdpa_fwd_fp8_workspace_size(ctypes.byref(p)))


def sdpa_fwd_fp8(q8, k8, v8, *, descale=(1.0, 1.0, 1.0), layout="bshd", mask="none", window=(-1, -1), scale=None,
                 cu_seqlens_q=None, cu_seqlens_kv=None, max_seqlen_q=None, max_seqlen_kv=None, out_dtype=None,
                 out=None, lse=None, workspace=None, stream=None):
    """FP8 E4M3 forward (head_dim 128 or 256). q8, k8, v8: torch.uint8 codes or
    torch.float8_e4m3fn tensors in `layout`; descale = (d_q, d_k, d_v), the
    per-tensor factors that turn codes into values. The softmax output is
    stored as E4M3(exp(S - m) * 448), m the row's final maximum, and O divides
    by 448 times the row sum (see sdpa_fwd_fp8 in include/sdpa.h). Returns (o, lse): o in out_dtype (default bfloat16) with
    q8's shape, lse float32 [rows_q, Hq]."""
    import torch

    f8 = getattr(torch, "float8_e4m3fn", None)
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.dtype not in (torch.uint8, f8):
            raise ValueError(f"{name} must hold E4M3 codes (torch.uint8 or torch.float8_e4m3fn), got {t.dtype}")
        if t.device != q8.device:
            raise ValueError(f"{name} must be on q8's device")
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    if out_dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("out_dtype must be bfloat16 or float16")
    rank = 3 if layout == "thd" else 4
    if any(t.dim() != rank for t in (q8, k8, v8)):
        raise ValueError(f"q8, k8, v8 must have {rank} dimensions in layout {layout}")
    if tuple(k8.shape) != tuple(v8.shape) or k8.shape[-1] != q8.shape[-1]:
        raise ValueError("k8 and v8 must have the same shape, and the same head_dim as q8")
    batch = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_problem(q8, k8, layout=layout, mask=mask, window=window, scale=scale, batch=batch,
                     dtype={torch.bfloat16: 0, torch.float16: 1}[out_dtype], max_seqlen_q=max_seqlen_q,
                     max_seqlen_kv=max_seqlen_kv)
    rows_q = q8.numel() // (q8.shape[-1] * q8.shape[-2])
    if out is None:
        out = torch.empty(tuple(q8.shape), dtype=out_dtype, device=q8.device)
    if lse is None:
        lse = torch.empty((rows_q, q8.shape[-2]), dtype=torch.float32, device=q8.device)
    if tuple(out.shape) != tuple(q8.shape) or out.dtype != out_dtype or tuple(lse.shape) != (rows_q, q8.shape[-2]) \
            or lse.dtype != torch.float32:
        raise ValueError("out must have q8's shape in out_dtype and lse float32 [rows_q, Hq]")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_kv", cu_seqlens_kv)):
        if t is not None and (t.dtype != torch.int32 or t.dim() != 1 or t.device != q8.device):
            raise ValueError(f"{name} must be a 1-D int32 tensor on q8's device")
    need = sdpa_fwd_fp8_workspace_size(p)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q8.device)
    _check_cuda(q8, k8, v8, out, lse, cu_seqlens_q, cu_seqlens_kv, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sdpa_fwd_fp8(ctypes.byref(p), _ptr(q8), _ptr(k8), _ptr(v8), float(descale[0]), float(descale[1]),
                            float(descale[2]), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
                            _ptr(workspace), ws_bytes, _stream(stream))
    if rc:
        raise SdpaError(rc, "sdpa_fwd_fp8")
    return out, lse


def sdpa_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return int(lib().sdpa_get_device_error(_stream(stream)))


def sdpa_debug_set_max_ctas(max_ctas: int) -> None:
    """Testing aid: cap the CTAs of every attention kernel launch (0 = no
    cap). See sdpa_debug_set_max_ctas in include/sdpa.h."""
    rc = lib().sdpa_debug_set_max_ctas(int(max_ctas))
    if rc:
        raise SdpaError(rc, "sdpa_debug_set_max_ctas")


def sdpa_last_launch_count() -> int:
    return int(lib().sdpa_last_launch_count())


def sdpa_profile_begin() -> None:
    """Start recording CUDA events around every kernel this thread's calls launch."""
    lib().sdpa_profile_begin()


def sdpa_profile_end() -> dict:
    """Stop recording; returns {kind: (total_ms, launches)} (synchronises)."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    rc = lib().sdpa_profile_end(ms, cnt, n)
    if rc:
        raise SdpaError(rc, "sdpa_profile_end")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def sdpa_merge(o_parts, lse_parts, *, out=None, lse=None, stream=None):
    """Log-sum-exp merge of partial results over a split of the keys.

    o_parts: [P, ..., H, D] (bf16/fp16, the forward's O over P key blocks,
    stacked); lse_parts: fp32 [P, rows, H] (the forward's LSE). Returns
    (o [..., H, D], lse [rows, H]).
    """
    import torch

    n = o_parts.shape[0]
    d = o_parts.shape[-1]
    items = o_parts[0].numel() // d
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    if lse_parts.dtype != torch.float32 or lse_parts.numel() != n * items or lse.numel() != items:
        raise ValueError("lse_parts must be float32 [P, rows, H] matching o_parts")
    if lse.dtype != torch.float32 or out.dtype != o_parts.dtype or out.numel() != items * d:
        raise ValueError("out must have o_parts' dtype and o_parts[0]'s size, lse must be float32 [rows, H]")
    if len({t.device for t in (o_parts, lse_parts, out, lse)}) != 1:
        raise ValueError("sdpa_merge tensors must be on one device")
    for t in (o_parts, lse_parts, out, lse):
        if not t.is_contiguous():
            raise ValueError("sdpa_merge needs contiguous tensors")
    _check_cuda(o_parts, lse_parts, out, lse)
    dt = {torch.bfloat16: 0, torch.float16: 1}.get(o_parts.dtype)
    if dt is None:
        raise ValueError("o_parts must be bf16 or fp16")
    p = MergeProblem(dt, items, d, n)
    rc = lib().sdpa_merge(ctypes.byref(p), _ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse), _stream(stream))
    if rc:
        raise SdpaError(rc, "sdpa_merge")
    return out, lse


def sdpa_selftest_bounded_wait(limit_us: int = 20000, stream=None) -> None:
    """Launch the bounded-wait self-test (records SDPA_ERR_TIMEOUT on the device)."""
    rc = lib().sdpa_selftest_bounded_wait(int(limit_us), _stream(stream))
    if rc:
        raise SdpaError(rc, "sdpa_selftest_bounded_wait")
