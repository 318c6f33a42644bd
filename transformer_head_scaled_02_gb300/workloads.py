"""Seeded synthetic inputs for the multi-head attention forward.

This module only draws random numbers, rounds them to the storage type and
counts work; it holds none of the attention arithmetic.  It is the one module
that both the CUDA path's callers (tests, bench) and the fp64 oracle's callers
use, so that the two sides always see bit-identical inputs.

Recipe (every workload):
  * generator: numpy ``default_rng(seed)`` (PCG64), seed 0 unless stated;
  * draw order, all in float32: X_q, X_kv (cross-attention only), W_qkv,
    b_qkv, W_o, b_o, kv_lengths (cross-attention with padding only);
  * bf16 workloads round every float tensor to bfloat16 with
    round-to-nearest-even; the rounded values are what both sides consume;
  * weights are (in, out) row-major: W_qkv is (D, 2*h*d_k + h*d_v) with column
    blocks [Q | K | V], W_o is (h*d_v, D).

The five named workloads are the shapes of the multi-head attention layer the
pages describe (itwiki.kr "멀티 헤드 어텐션": d_model 512, h 8, d_k 64 as in the
original paper; molayo1419.me "MHA란 무엇인가?": E = 512, h = 8; the
greeksharifa.github.io summary of Multi-Token Attention, appendix D: an 880M
model with width 1536, 16 heads and context 2048), at sizes a GB300 works on.
No dataset, checkpoint or trained weight is involved anywhere.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T_q: int
    T_kv: int
    D: int
    h: int
    d_k: int
    d_v: int
    dtype: str            # "f32" or "bf16": storage type of every tensor
    causal: bool
    cross: bool           # K, V from a second state tensor X_kv
    weight_init: str      # "uniform_inv_sqrt_d" | "xavier_uniform" | "normal_0.02"
    bias: str             # "uniform_0.1" | "zero" | "normal_0.02" | "none"
    kv_len_range: Optional[tuple] = None   # inclusive (lo, hi) for per-batch valid key lengths
    description: str = ""

    @property
    def w_cols(self) -> int:
        return 2 * self.h * self.d_k + self.h * self.d_v


WORKLOADS = {
    "c1_f32_tiny": Workload(
        "c1_f32_tiny", B=1, T_q=16, T_kv=16, D=32, h=8, d_k=4, d_v=4, dtype="f32",
        causal=False, cross=False, weight_init="uniform_inv_sqrt_d", bias="uniform_0.1",
        description="self-attention, fp32, non-causal, B=1 T=16 D=32 h=8 d=4"),
    "c2_f32_causal": Workload(
        "c2_f32_causal", B=8, T_q=128, T_kv=128, D=512, h=8, d_k=64, d_v=64, dtype="f32",
        causal=True, cross=False, weight_init="xavier_uniform", bias="zero",
        description="self-attention, fp32, causal, B=8 T=128 D=512 h=8 d=64"),
    "c3_bf16_causal": Workload(
        "c3_bf16_causal", B=4, T_q=2048, T_kv=2048, D=1024, h=16, d_k=64, d_v=64, dtype="bf16",
        causal=True, cross=False, weight_init="normal_0.02", bias="normal_0.02",
        description="self-attention, bf16 storage / fp32 accumulate, causal, B=4 T=2048 D=1024 h=16 d=64"),
    "c4_bf16_causal_long": Workload(
        "c4_bf16_causal_long", B=1, T_q=16384, T_kv=16384, D=2048, h=16, d_k=128, d_v=128,
        dtype="bf16", causal=True, cross=False, weight_init="normal_0.02", bias="none",
        description="long-sequence self-attention, bf16, causal, B=1 T=16384 D=2048 h=16 d=128"),
    "c5_bf16_cross": Workload(
        "c5_bf16_cross", B=16, T_q=512, T_kv=4096, D=768, h=12, d_k=64, d_v=64, dtype="bf16",
        causal=False, cross=True, weight_init="normal_0.02", bias="none",
        kv_len_range=(1024, 4096),
        description="encoder-decoder cross-attention, bf16, non-causal, B=16 T_q=512 "
                    "T_kv=4096 D=768 h=12 d=64, valid key lengths U{1024..4096}"),
}


def custom(name: str, B: int, T_q: int, D: int, h: int, d_k: int, d_v: Optional[int] = None,
           T_kv: Optional[int] = None, dtype: str = "bf16", causal: bool = False,
           cross: bool = False, weight_init: str = "normal_0.02", bias: str = "normal_0.02",
           kv_len_range: Optional[tuple] = None) -> Workload:
    """A workload of any shape, drawn with the same recipe as the named ones."""
    return Workload(name, B=B, T_q=T_q, T_kv=T_q if T_kv is None else T_kv, D=D, h=h,
                    d_k=d_k, d_v=d_k if d_v is None else d_v, dtype=dtype, causal=causal,
                    cross=cross, weight_init=weight_init, bias=bias, kv_len_range=kv_len_range)


# --------------------------------------------------------------------------
# bfloat16 storage rounding (round-to-nearest-even on the float32 bit pattern)
# --------------------------------------------------------------------------

def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values rounded to bfloat16 (RNE).
    NaN stays a quiet NaN; infinities and signed zeros are kept."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    rounded = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    nan = np.isnan(a)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """float32 values of bfloat16 bit patterns (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 array holding the bfloat16-rounded values of ``a``."""
    return bf16_to_f32(bf16_bits(a))


# --------------------------------------------------------------------------
# drawing
# --------------------------------------------------------------------------

def _weights(rng, shape, init: str, fan_in: int, fan_out: int) -> np.ndarray:
    if init == "uniform_inv_sqrt_d":
        a = 1.0 / math.sqrt(fan_in)
        return rng.uniform(-a, a, size=shape).astype(np.float32)
    if init == "xavier_uniform":
        a = math.sqrt(6.0 / (fan_in + fan_out))
        return rng.uniform(-a, a, size=shape).astype(np.float32)
    if init == "normal_0.02":
        return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(0.02)
    raise ValueError(f"unknown weight init {init!r}")


def _bias(rng, n: int, kind: str) -> Optional[np.ndarray]:
    if kind == "none":
        return None
    if kind == "zero":
        return np.zeros(n, dtype=np.float32)
    if kind == "uniform_0.1":
        return rng.uniform(-0.1, 0.1, size=n).astype(np.float32)
    if kind == "normal_0.02":
        return rng.standard_normal(size=n, dtype=np.float32) * np.float32(0.02)
    raise ValueError(f"unknown bias kind {kind!r}")


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw every input of workload ``w``.  Returns float32 arrays (bf16-rounded
    for bf16 workloads) and int32 kv_lengths (or None):
    keys X_q, X_kv (None for self-attention), W_qkv, b_qkv, W_o, b_o, kv_lengths."""
    rng = np.random.default_rng(seed)
    X_q = rng.standard_normal(size=(w.B, w.T_q, w.D), dtype=np.float32)
    X_kv = rng.standard_normal(size=(w.B, w.T_kv, w.D), dtype=np.float32) if w.cross else None
    # The fused (D, 3D) projection is treated as one tensor for Xavier: fan_in D,
    # fan_out w_cols; W_o has fan_in h*d_v and fan_out D.
    W_qkv = _weights(rng, (w.D, w.w_cols), w.weight_init, w.D, w.w_cols)
    b_qkv = _bias(rng, w.w_cols, w.bias)
    W_o = _weights(rng, (w.h * w.d_v, w.D), w.weight_init, w.h * w.d_v, w.D)
    b_o = _bias(rng, w.D, w.bias)
    kv_lengths = None
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        kv_lengths = rng.integers(lo, hi, size=w.B, endpoint=True).astype(np.int32)
    out = dict(X_q=X_q, X_kv=X_kv, W_qkv=W_qkv, b_qkv=b_qkv, W_o=W_o, b_o=b_o,
               kv_lengths=kv_lengths)
    if w.dtype == "bf16":
        for k in ("X_q", "X_kv", "W_qkv", "b_qkv", "W_o", "b_o"):
            if out[k] is not None:
                out[k] = round_to_bf16(out[k])
    elif w.dtype != "f32":
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return out


# --------------------------------------------------------------------------
# work accounting
# --------------------------------------------------------------------------

def flops(w: Workload, kv_lengths=None) -> dict:
    """FLOPs of one forward, counting a multiply-add as 2 (itwiki.kr
    "멀티 헤드 어텐션", 매개변수와 계산량: about 8 T D^2 for the four projections
    and 4 T^2 D for scores plus weighted sum).  Causal masking halves the
    attention term.  Cross-attention: projections 4 T_q D^2 + 4 T_kv D^2,
    attention 4 T_q T_kv D.  ``alg_*`` replaces T_kv by each batch's valid
    length L_b (padded keys need neither projection nor attention)."""
    D, B = w.D, w.B
    half = 0.5 if w.causal else 1.0
    proj = B * (4.0 * w.T_q * D * D + 4.0 * w.T_kv * D * D)
    attn = B * 4.0 * w.T_q * w.T_kv * D * half
    out = {"proj": proj, "attn": attn, "total": proj + attn}
    if kv_lengths is not None:
        L = np.asarray(kv_lengths, dtype=np.float64)
        ap = B * 4.0 * w.T_q * D * D + float(np.sum(4.0 * L * D * D))
        aa = float(np.sum(4.0 * w.T_q * L * D)) * half
        out.update(alg_proj=ap, alg_attn=aa, alg_total=ap + aa)
    return out


def step_flops(w: Workload) -> dict:
    """Per-kernel FLOPs as the three launches compute them (2 per multiply-add):
    the Q/K/V projection GEMM(s), the fused attention (causal: only the lower
    triangle counted), and the output projection GEMM."""
    hq, hv = w.h * w.d_k, w.h * w.d_v
    qkv = 2.0 * w.B * (w.T_q * w.D * hq + w.T_kv * w.D * (hq + hv))
    half = 0.5 if w.causal else 1.0
    attn = 2.0 * w.B * w.h * w.T_q * w.T_kv * (w.d_k + w.d_v) * half
    out = 2.0 * w.B * w.T_q * hv * w.D
    return {"qkv_proj": qkv, "attention": attn, "out_proj": out}


def hbm_bytes(w: Workload) -> float:
    """Algorithmic HBM bytes of the unfused-GEMM / fused-attention path: read X
    (and X_kv), write then read Q, K, V, write then read Ocat, write Y, read each
    weight once.  The (B,h,T,T) scores never move."""
    s = 4 if w.dtype == "f32" else 2
    hq, hv = w.h * w.d_k, w.h * w.d_v
    x = w.B * w.T_q * w.D + (w.B * w.T_kv * w.D if w.cross else 0)
    qkv = w.B * w.T_q * hq + w.B * w.T_kv * (hq + hv)
    ocat = w.B * w.T_q * hv
    y = w.B * w.T_q * w.D
    weights = w.D * w.w_cols + hv * w.D + w.w_cols + w.D
    return float(s * (x + 2 * qkv + 2 * ocat + y + weights))


def random_tensor(shape, seed: int, dtype: str = "bf16", scale: float = 1.0) -> np.ndarray:
    """A standalone N(0, scale^2) tensor (float32, bf16-rounded for "bf16"), for
    tests of a single step (projection or attention) on given operands."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)
    return round_to_bf16(a) if dtype == "bf16" else a
