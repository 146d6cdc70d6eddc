"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random inputs and describes their shapes; it holds none
of the attention arithmetic, so the oracle and the CUDA path can both be fed
from it without sharing any computation.

Draw order for every workload (one numpy PCG64 stream per seed): the varlen
lengths (THD only), then q, k, v, dO, each as float64 N(0, 1) * std. The
float64 arrays are the masters; the kernel and the oracle both consume the
same dtype-rounded copies (rounded through float32, round-to-nearest-even).

Workload shapes follow the pages' workloads: D128 BF16 causal compact THD with
Hq32/Hkv8 (TransformerEngine PR #3705), b2 hq8 hkv4 d512 causal (PR #3527,
"Performance"), and sliding-window D256 layers (PR #3527, "Problem"). The
asymmetric forward (Q/K 192, V/O 128: PR #3527, "Scope", the forward engine's
native (192, 128) shape) reuses the compact THD workload's lengths and heads,
since the pages give no workload of its own.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layout: str          # "bshd" | "sbhd" | "thd"
    mask: str            # "none" | "causal" | "causal_br"
    batch: int
    seqlen_q: int        # THD: the largest length allowed by `len_range`
    seqlen_kv: int
    heads_q: int
    heads_kv: int
    head_dim: int
    dtype: str           # "bf16" | "fp16"
    window: tuple = (-1, -1)
    std: float = 1.0
    len_range: tuple | None = None  # THD: inclusive (lo, hi) of the uniform lengths
    head_dim_v: int = 0             # width of V, O and dO rows; 0 = head_dim

    @property
    def dv(self) -> int:
        return self.head_dim_v or self.head_dim

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY = Workload("tiny", "bshd", "causal", 1, 128, 128, 2, 2, 128, "bf16")
VARLEN_THD = Workload("varlen_thd_gqa", "thd", "causal", 8, 4096, 4096, 32, 8, 128, "bf16", len_range=(512, 4096))
SLIDING = Workload("sliding_window_d256", "bshd", "causal", 2, 8192, 8192, 16, 8, 256, "bf16", window=(1024, 0))
D512_BR = Workload("d512_rect_bottom_right", "bshd", "causal_br", 2, 2048, 8192, 16, 4, 512, "bf16")
D512_NC = Workload("d512_rect_noncausal", "bshd", "none", 2, 2048, 8192, 16, 4, 512, "bf16")
LONG_FP16 = Workload("long_context_fp16_sbhd", "sbhd", "causal", 1, 32768, 32768, 16, 16, 128, "fp16", std=0.5)
# forward only (the backward requires d_qk == d_v)
ASYM = Workload("varlen_thd_gqa_d192_v128", "thd", "causal", 8, 4096, 4096, 32, 8, 192, "bf16", len_range=(512, 4096),
                head_dim_v=128)

ALL = [TINY, VARLEN_THD, SLIDING, D512_BR, D512_NC, LONG_FP16, ASYM]
FORWARD_ONLY = {ASYM.name}
SEEDS = {"tiny": 1000, "varlen_thd_gqa": 1001, "sliding_window_d256": 1002, "d512_rect_bottom_right": 1003,
         "d512_rect_noncausal": 1003, "long_context_fp16_sbhd": 1004, "varlen_thd_gqa_d192_v128": 1001}


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to bf16/fp16 (through float32, RNE); returns float64."""
    import torch

    td = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(td).to(torch.float64).numpy()


def to_torch(x: np.ndarray, dtype: str):
    """float64 numpy -> CPU torch tensor of the storage dtype."""
    import torch

    td = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(td)


def shapes(w: Workload, lengths_q=None, lengths_kv=None, d_q=None, d_kv=None):
    """(q-side shape, kv-side shape); the last dimensions default to head_dim."""
    d_q = w.head_dim if d_q is None else d_q
    d_kv = w.head_dim if d_kv is None else d_kv
    if w.layout == "bshd":
        return (w.batch, w.seqlen_q, w.heads_q, d_q), (w.batch, w.seqlen_kv, w.heads_kv, d_kv)
    if w.layout == "sbhd":
        return (w.seqlen_q, w.batch, w.heads_q, d_q), (w.seqlen_kv, w.batch, w.heads_kv, d_kv)
    return (int(np.sum(lengths_q)), w.heads_q, d_q), (int(np.sum(lengths_kv)), w.heads_kv, d_kv)


def _draw_lengths(w: Workload, rng) -> np.ndarray:
    lo, hi = w.len_range if w.len_range else (1, w.seqlen_q)
    return rng.integers(lo, hi + 1, size=w.batch)


def thd_lengths(w: Workload, seed: int | None = None) -> np.ndarray:
    """The per-sequence lengths make_inputs draws for a THD workload (the
    first draw of its stream), without drawing the tensors."""
    seed = SEEDS.get(w.name, 0) if seed is None else seed
    return _draw_lengths(w, np.random.Generator(np.random.PCG64(seed)))


def make_inputs(w: Workload, seed: int | None = None, lengths=None):
    """Draw the float64 masters. Returns a dict with q, k, v, do and, for THD,
    cu_seqlens_q / cu_seqlens_kv (int32, zero-based cumulative, B+1 entries).

    `lengths` (THD) overrides the drawn lengths: an int array, or a pair
    (lengths_q, lengths_kv).
    """
    seed = SEEDS.get(w.name, 0) if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    lq = lk = None
    if w.layout == "thd":
        drawn = _draw_lengths(w, rng)
        if lengths is None:
            lq = lk = drawn
        elif isinstance(lengths, tuple):
            lq, lk = np.asarray(lengths[0]), np.asarray(lengths[1])
        else:
            lq = lk = np.asarray(lengths)
        out["cu_seqlens_q"] = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        out["cu_seqlens_kv"] = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    sq, sk = shapes(w, lq, lk)
    so, sv = shapes(w, lq, lk, w.dv, w.dv)  # O/dO and V rows are head_dim_v wide
    out["q"] = rng.standard_normal(sq) * w.std
    out["k"] = rng.standard_normal(sk) * w.std
    out["v"] = rng.standard_normal(sv) * w.std
    out["do"] = rng.standard_normal(so) * w.std
    return out


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8, the finite-only OCP format) nearest to float64
    values, through torch's float8_e4m3fn conversion (round to nearest even,
    saturating): the FP8 inputs are these codes of seeded normal masters."""
    import torch

    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


FP8_STD = 3.0                     # the codes' masters are N(0, 1) * 3 (a spread over most of E4M3's range)
FP8_DESCALE = (0.5, 0.25, 0.125)  # per-tensor descales of Q, K, V


def fp8_inputs(w: Workload, seed: int | None = None, lengths=None) -> dict:
    """make_inputs' draws for `w`, each master times FP8_STD, as E4M3 codes
    q8, k8, v8 (cu_seqlens copied); dO is not drawn into codes."""
    inp = make_inputs(w, seed=seed, lengths=lengths)
    out = {key: val for key, val in inp.items() if key.startswith("cu_")}
    for key in ("q", "k", "v"):
        out[key + "8"] = e4m3_codes(inp[key] * FP8_STD)
    return out


def rounded(inputs: dict, dtype: str) -> dict:
    """The dtype-rounded copies (as float64) of q, k, v, do; other keys copied."""
    out = dict(inputs)
    for key in ("q", "k", "v", "do"):
        out[key] = round_to(inputs[key], dtype)
    return out
