"""Python binding of the float64 CPU attention oracle (``sdpa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it. The CUDA product path never imports this module and
shares no code with it.

Arrays are numpy float64 in the caller's layout:
  "bshd": (B, S, H, D)    "sbhd": (S, B, H, D)    "thd": (T, H, D)
LSE and delta are token-major (rows_q, Hq), rows in Q's leading order.
Masks: "none", "causal" (top-left), "causal_br" (bottom-right).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libsdpa_oracle.so")

LAYOUTS = {"bshd": 0, "sbhd": 1, "thd": 2}
MASKS = {"none": 0, "causal": 1, "causal_br": 2}

_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int),
        ("mask_type", ctypes.c_int),
        ("batch", ctypes.c_int),
        ("seqlen_q", ctypes.c_int),
        ("seqlen_kv", ctypes.c_int),
        ("num_heads_q", ctypes.c_int),
        ("num_heads_kv", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("window_left", ctypes.c_int),
        ("window_right", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("head_dim_v", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, OpenMP) into oracle/_build."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            pp = ctypes.POINTER(_Problem)
            lib.sdpa_oracle_fwd.argtypes = [pp, dp, dp, dp, ip, ip, dp, dp]
            lib.sdpa_oracle_fwd_rows.argtypes = [pp, dp, dp, dp, ip, ip, ctypes.c_int, ip, dp, dp]
            lib.sdpa_oracle_bwd_part.argtypes = [pp, dp, dp, dp, dp, ip, ip, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, dp]
            lib.sdpa_oracle_dq_rows.argtypes = [pp, dp, dp, dp, dp, ip, ip, ctypes.c_int, ip, dp]
            lib.sdpa_oracle_dkdv_rows.argtypes = [pp, dp, dp, dp, dp, ip, ip, ctypes.c_int, ip, dp, dp]
            lib.sdpa_oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, dp, dp, dp, dp]
            u8p = ctypes.POINTER(ctypes.c_uint8)
            dbl = ctypes.c_double
            lib.sdpa_oracle_fwd_fp8.argtypes = [pp, u8p, u8p, u8p, dbl, dbl, dbl, dbl, ip, ip, dp, dp]
            lib.sdpa_oracle_e4m3_round_array.argtypes = [ctypes.c_int64, dp, dp]
            lib.sdpa_oracle_e4m3_decode_array.argtypes = [ctypes.c_int64, u8p, dp]
            lib.sdpa_oracle_num_threads.restype = ctypes.c_int
            lib.sdpa_oracle_probs.argtypes = [pp, dp, dp, ip, ip, dp]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().sdpa_oracle_num_threads())


def _dptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    if a is None:
        return None
    assert a.dtype == np.int32 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class Problem:
    """Geometry of one attention call, inferred from the array shapes."""

    def __init__(self, q, k, layout, mask, scale, window=(-1, -1), cu_q=None, cu_kv=None, v=None):
        self.layout = layout
        self.mask = mask
        if layout == "bshd":
            self.batch, self.sq, self.hq, self.d = q.shape
            self.sk, self.hkv = k.shape[1], k.shape[2]
        elif layout == "sbhd":
            self.sq, self.batch, self.hq, self.d = q.shape
            self.sk, self.hkv = k.shape[0], k.shape[2]
        elif layout == "thd":
            assert cu_q is not None and cu_kv is not None
            self.batch = len(cu_q) - 1
            self.hq, self.d = q.shape[1], q.shape[2]
            self.hkv = k.shape[1]
            self.sq = int(np.max(np.diff(cu_q))) if self.batch else 0
            self.sk = int(np.max(np.diff(cu_kv))) if self.batch else 0
        else:
            raise ValueError(layout)
        self.rows_q = q.shape[0] * (q.shape[1] if layout != "thd" else 1)
        self.rows_kv = k.shape[0] * (k.shape[1] if layout != "thd" else 1)
        self.cu_q = None if cu_q is None else np.ascontiguousarray(cu_q, dtype=np.int32)
        self.cu_kv = None if cu_kv is None else np.ascontiguousarray(cu_kv, dtype=np.int32)
        # width of v and o rows (the forward allows it to differ from q/k's)
        self.dv = self.d if v is None else v.shape[-1]
        self.c = _Problem(LAYOUTS[layout], MASKS[mask], self.batch, self.sq if layout != "thd" else 0,
                          self.sk if layout != "thd" else 0, self.hq, self.hkv, self.d, int(window[0]),
                          int(window[1]), float(scale), self.dv)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def fwd(q, k, v, *, layout="bshd", mask="none", scale=None, window=(-1, -1), cu_q=None, cu_kv=None):
    """Full forward. Returns (o, lse): o in Q's layout with V's last dimension
    (which may differ from Q/K's), lse (rows_q, Hq)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    p = Problem(q, k, layout, mask, scale, window, cu_q, cu_kv, v=v)
    o = np.zeros(q.shape[:-1] + (p.dv,))
    lse = np.full((p.rows_q, p.hq), -np.inf)
    rc = _load().sdpa_oracle_fwd(ctypes.byref(p.c), _dptr(q), _dptr(k), _dptr(v), _iptr(p.cu_q), _iptr(p.cu_kv),
                                 _dptr(o), _dptr(lse))
    if rc:
        raise ValueError(f"oracle fwd rejected the problem (rc={rc})")
    return o, lse


def bwd(q, k, v, dout, *, layout="bshd", mask="none", scale=None, window=(-1, -1), cu_q=None, cu_kv=None,
        batch_range=None, kv_head_range=None):
    """Backward from the inputs alone. Returns dict with dq, dk, dv, o, lse, delta.

    batch_range / kv_head_range restrict the work (rows outside stay zero).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    p = Problem(q, k, layout, mask, scale, window, cu_q, cu_kv, v=v)
    b0, b1 = batch_range or (0, p.batch)
    g0, g1 = kv_head_range or (0, p.hkv)
    out = {
        "dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "o": np.zeros_like(q),
        "lse": np.full((p.rows_q, p.hq), -np.inf), "delta": np.zeros((p.rows_q, p.hq)),
    }
    rc = _load().sdpa_oracle_bwd_part(ctypes.byref(p.c), _dptr(q), _dptr(k), _dptr(v), _dptr(dout), _iptr(p.cu_q),
                                      _iptr(p.cu_kv), b0, b1, g0, g1, _dptr(out["dq"]), _dptr(out["dk"]),
                                      _dptr(out["dv"]), _dptr(out["o"]), _dptr(out["lse"]), _dptr(out["delta"]))
    if rc:
        raise ValueError(f"oracle bwd rejected the problem (rc={rc})")
    return out


def fwd_rows(q, k, v, bhi, *, layout="bshd", mask="none", scale=None, window=(-1, -1), cu_q=None, cu_kv=None):
    """Forward for selected (b, h, i) rows. Returns (o_rows (n, Dv), lse_rows (n,))."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    p = Problem(q, k, layout, mask, scale, window, cu_q, cu_kv, v=v)
    bhi = np.ascontiguousarray(bhi, dtype=np.int32).reshape(-1, 3)
    o = np.zeros((len(bhi), p.dv))
    lse = np.zeros(len(bhi))
    rc = _load().sdpa_oracle_fwd_rows(ctypes.byref(p.c), _dptr(q), _dptr(k), _dptr(v), _iptr(p.cu_q),
                                      _iptr(p.cu_kv), len(bhi), _iptr(bhi), _dptr(o), _dptr(lse))
    if rc:
        raise ValueError(f"oracle fwd_rows rejected the problem (rc={rc})")
    return o, lse


def dq_rows(q, k, v, dout, bhi, *, layout="bshd", mask="none", scale=None, window=(-1, -1), cu_q=None,
            cu_kv=None):
    """dQ for selected (b, h, i) rows. Returns (n, D)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    p = Problem(q, k, layout, mask, scale, window, cu_q, cu_kv, v=v)
    bhi = np.ascontiguousarray(bhi, dtype=np.int32).reshape(-1, 3)
    dq = np.zeros((len(bhi), p.d))
    rc = _load().sdpa_oracle_dq_rows(ctypes.byref(p.c), _dptr(q), _dptr(k), _dptr(v), _dptr(dout), _iptr(p.cu_q),
                                     _iptr(p.cu_kv), len(bhi), _iptr(bhi), _dptr(dq))
    if rc:
        raise ValueError(f"oracle dq_rows rejected the problem (rc={rc})")
    return dq


def dkdv_rows(q, k, v, dout, bgj, *, layout="bshd", mask="none", scale=None, window=(-1, -1), cu_q=None,
              cu_kv=None):
    """dK and dV for selected (b, kv head g, key j) rows. Returns (dk (n, D), dv (n, D))."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    p = Problem(q, k, layout, mask, scale, window, cu_q, cu_kv, v=v)
    bgj = np.ascontiguousarray(bgj, dtype=np.int32).reshape(-1, 3)
    dk = np.zeros((len(bgj), p.d))
    dv = np.zeros((len(bgj), p.d))
    rc = _load().sdpa_oracle_dkdv_rows(ctypes.byref(p.c), _dptr(q), _dptr(k), _dptr(v), _dptr(dout), _iptr(p.cu_q),
                                       _iptr(p.cu_kv), len(bgj), _iptr(bgj), _dptr(dk), _dptr(dv))
    if rc:
        raise ValueError(f"oracle dkdv_rows rejected the problem (rc={rc})")
    return dk, dv


def probs(q, k, *, layout="bshd", mask="none", scale=None, window=(-1, -1), cu_q=None, cu_kv=None):
    """Softmax probabilities p_ij = exp(s_ij - LSE_i) of every query row:
    array (rows_q, Hq, lk_max), zero at masked keys and past a sequence's
    keys (lk_max = the longest key sequence)."""
    q, k = _f64(q), _f64(k)
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    p = Problem(q, k, layout, mask, scale, window, cu_q, cu_kv)
    out = np.zeros((p.rows_q, p.hq, max(p.sk, 1)))
    rc = _load().sdpa_oracle_probs(ctypes.byref(p.c), _dptr(q), _dptr(k), _iptr(p.cu_q), _iptr(p.cu_kv), _dptr(out))
    if rc:
        raise ValueError(f"oracle probs rejected the problem (rc={rc})")
    return out


def merge(o_parts, lse_parts):
    """Combine partial results over a split of the keys (log-sum-exp merge).

    o_parts (P, ..., D) and lse_parts (P, ...) with the same middle shape;
    returns (o (..., D), lse (...)). Empty blocks carry lse = -inf.
    """
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    n = o_parts.shape[0]
    d = o_parts.shape[-1]
    mid = o_parts.shape[1:-1]
    assert lse_parts.shape == (n,) + mid
    items = int(np.prod(mid)) if mid else 1
    o = np.zeros(mid + (d,))
    lse = np.zeros(mid)
    rc = _load().sdpa_oracle_merge(n, items, d, _dptr(o_parts), _dptr(lse_parts), _dptr(o), _dptr(lse))
    if rc:
        raise ValueError(f"oracle merge rejected the problem (rc={rc})")
    return o, lse


# ---------------------------------------------------------------- FP8 E4M3
def _u8ptr(a):
    assert a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def e4m3_decode(codes):
    """Real values of E4M3 codes (uint8 array), NaN for the NaN codes."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape)
    _load().sdpa_oracle_e4m3_decode_array(c.size, _u8ptr(c), _dptr(out))
    return out


def e4m3_round(x):
    """Nearest E4M3 values (ties to even; |x| >= 448 saturates to 448)."""
    x = _f64(x)
    out = np.zeros(x.shape)
    _load().sdpa_oracle_e4m3_round_array(x.size, _dptr(x), _dptr(out))
    return out


def fwd_fp8(q8, k8, v8, *, descale=(1.0, 1.0, 1.0), scale_s=448.0, layout="bshd", mask="none", scale=None,
            window=(-1, -1), cu_q=None, cu_kv=None):
    """FP8 E4M3 forward: q8/k8/v8 are E4M3 codes (uint8) in their layouts with
    per-tensor descales (d_q, d_k, d_v); the softmax output normalised by its
    row maximum is stored as P8 = E4M3(exp(s - m) * scale_s) and
    O = P8 V * d_v / (scale_s * sum_j exp(s_j - m)). Returns (o, lse) like fwd."""
    q8, k8, v8 = (np.ascontiguousarray(x, dtype=np.uint8) for x in (q8, k8, v8))
    scale = 1.0 / np.sqrt(q8.shape[-1]) if scale is None else scale
    p = Problem(q8, k8, layout, mask, scale, window, cu_q, cu_kv, v=v8)
    o = np.zeros(q8.shape[:-1] + (p.dv,))
    lse = np.full((p.rows_q, p.hq), -np.inf)
    rc = _load().sdpa_oracle_fwd_fp8(ctypes.byref(p.c), _u8ptr(q8), _u8ptr(k8), _u8ptr(v8), float(descale[0]),
                                     float(descale[1]), float(descale[2]), float(scale_s), _iptr(p.cu_q),
                                     _iptr(p.cu_kv), _dptr(o), _dptr(lse))
    if rc:
        raise ValueError(f"oracle fwd_fp8 rejected the problem (rc={rc})")
    return o, lse
