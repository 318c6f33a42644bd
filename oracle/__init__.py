"""fp64 CPU oracle for the multi-head attention forward -- TEST INFRASTRUCTURE.

This package is the checker the CUDA path is compared against.  Only the test
suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import it.  The library in ``transformer_head_scaled_02_gb300`` never imports,
links or calls anything here, and the two share no code.

The arithmetic lives in ``mha_oracle.c`` (plain fp64 loops, OpenMP over
independent rows / (batch, head) pairs); this module only marshals numpy
arrays into it.  Every function converts its inputs to contiguous float64
first, so callers may hand in float32 arrays holding bf16-rounded values: the
conversion to fp64 is exact.

Sources followed (page title, section):
  * itwiki.kr "멀티 헤드 어텐션" -- 수식 (scaled dot-product attention and the
    multi-head composition) and 텐서 모양으로 본 계산 (the shape table: fused
    D x 3D projection, view+transpose head split, (B,h,T,T) scores, softmax over
    the last axis, Concat, W^O);
  * iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산" -- sections 9-10
    (causal mask as -inf, row softmax) and 19 (cross-attention);
  * molayo1419.me "MHA란 무엇인가?" -- key padding, and the all-masked row that
    comes out NaN.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mha_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile mha_oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_linear.restype = ctypes.c_int
            lib.oracle_linear.argtypes = [
                ctypes.c_long, ctypes.c_long, ctypes.c_long,
                _dp, ctypes.c_long, _dp, ctypes.c_long, _dp, _dp, ctypes.c_long,
                ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int,
                _dp, ctypes.c_long, _dp, ctypes.c_long, _dp, ctypes.c_long,
                ctypes.c_int, _ip, _ip, ctypes.c_int, _dp, ctypes.c_long, _dp,
                ctypes.c_int]
            lib.oracle_mha_forward.restype = ctypes.c_int
            lib.oracle_mha_forward.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _dp, _dp, _dp, _dp, _dp, _dp,
                ctypes.c_int, _ip, _ip, ctypes.c_int, _dp, ctypes.c_int]
            lib.oracle_attention_grouped.restype = ctypes.c_int
            lib.oracle_attention_grouped.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int,
                _dp, ctypes.c_long, _dp, ctypes.c_long, _dp, ctypes.c_long,
                ctypes.c_int, _ip, _ip, ctypes.c_int, _dp, ctypes.c_long, _dp,
                ctypes.c_int]
            lib.oracle_mha_forward_ex.restype = ctypes.c_int
            lib.oracle_mha_forward_ex.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                ctypes.c_int, _ip, _ip, ctypes.c_int, _dp, ctypes.c_int]
            lib.oracle_mha_forward_rounded.restype = ctypes.c_int
            lib.oracle_mha_forward_rounded.argtypes = lib.oracle_mha_forward_ex.argtypes
            lib.oracle_round_bf16.restype = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int,
                _dp, ctypes.c_long, _dp, ctypes.c_long, _dp, ctypes.c_long,
                _ip, _dp, ctypes.c_long, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _iptr(a):
    return None if a is None else a.ctypes.data_as(_ip)


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use by default."""
    return int(_load().oracle_max_threads())


def linear(X, W, b=None, nthreads: int = 0):
    """Y = X W + b for X (..., K), W (K, N), b (N) or None; fp64 result."""
    lib = _load()
    X = _f64(X)
    W = _f64(W)
    b = _f64(b)
    K, N = W.shape
    lead = X.shape[:-1]
    X2 = X.reshape(-1, K)
    M = X2.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_linear(M, K, N, _ptr(X2), K, _ptr(W), N, _ptr(b), _ptr(Y), N, nthreads)
    if rc:
        raise ValueError(f"oracle_linear failed ({rc})")
    return Y.reshape(*lead, N)


def attention(Q, K, V, h: int, causal: bool = False, kv_lengths=None, rows=None,
              return_weights: bool = False, nthreads: int = 0, h_kv=None):
    """Attention of every head over already-projected Q (B,Tq,h*dk),
    K (B,Tkv,h_kv*dk), V (B,Tkv,h_kv*dv) (h_kv = h unless given: grouped K/V heads,
    query head i using K/V head i // (h // h_kv)).  Returns Ocat (B, n_out, h*dv) --
    the Concat of the heads -- and, if asked, the weights (B, h, n_out, Tkv)."""
    lib = _load()
    Q = _f64(Q)
    K = _f64(K)
    V = _f64(V)
    h_kv = h if h_kv is None else int(h_kv)
    B, Tq, hdk = Q.shape
    _, Tkv, kvw = V.shape
    if hdk % h or kvw % h_kv or h % h_kv:
        raise ValueError("head counts do not divide the projection widths")
    dk, dv = hdk // h, kvw // h_kv
    if K.shape[2] != h_kv * dk:
        raise ValueError("K width is not h_kv * d_k")
    hdv = h * dv
    kvl = _i32(kv_lengths)
    rws = _i32(rows)
    n_out = Tq if rws is None else len(rws)
    O = np.empty((B, n_out, hdv), dtype=np.float64)
    P = np.empty((B, h, n_out, Tkv), dtype=np.float64) if return_weights else None
    rc = lib.oracle_attention_grouped(B, Tq, Tkv, h, h_kv, dk, dv, _ptr(Q), hdk, _ptr(K), h_kv * dk,
                                      _ptr(V), kvw, int(bool(causal)), _iptr(kvl), _iptr(rws),
                                      0 if rws is None else len(rws), _ptr(O), hdv, _ptr(P),
                                      nthreads)
    if rc:
        raise ValueError(f"oracle_attention failed ({rc})")
    return (O, P) if return_weights else O


def proj_width(h: int, d_k: int, d_v: int, h_kv=None, gated: bool = False) -> int:
    """Columns of the fused projection: [Q | K | V (| G)]."""
    h_kv = h if h_kv is None else int(h_kv)
    return h * d_k + h_kv * d_k + h_kv * d_v + (h * d_v if gated else 0)


def round_bf16(x: float) -> float:
    """x rounded to the nearest bfloat16 value, ties to even (the oracle's own rounding)."""
    return float(_load().oracle_round_bf16(float(x)))


def mha_forward(Xq, Wqkv, bqkv, Wo, bo, h: int, d_k: int, d_v: int, Xkv=None,
                causal: bool = False, kv_lengths=None, rows=None, nthreads: int = 0,
                h_kv=None, gated: bool = False, residual=None, round_bf16: bool = False):
    """The whole forward.  Xq (B,Tq,D); Xkv (B,Tkv,D) or None (self-attention);
    Wqkv (D, proj_width(...)) with column blocks [Q|K|V(|G)]; Wo (h*d_v, D).
    h_kv: K/V heads (default h); gated: sigmoid output gate from the G block;
    residual: (B,Tq,D) added to Y.  rows: optional query-row indices (shared by every
    batch) to compute.  round_bf16: the secondary diagnostic mode that rounds to bf16
    where the bf16 GPU path stores values (Q/K/V/G, the softmax weights entering the
    weighted sum, the attention output, Y).  Returns Y (B, n_out, D) in fp64."""
    lib = _load()
    Xq = _f64(Xq)
    Xkv = _f64(Xkv)
    Wqkv = _f64(Wqkv)
    bqkv = _f64(bqkv)
    Wo = _f64(Wo)
    bo = _f64(bo)
    R = _f64(residual)
    h_kv = h if h_kv is None else int(h_kv)
    B, Tq, D = Xq.shape
    Tkv = Tq if Xkv is None else Xkv.shape[1]
    if Wqkv.shape != (D, proj_width(h, d_k, d_v, h_kv, gated)) or Wo.shape != (h * d_v, D):
        raise ValueError("weight shapes do not match (D, h, h_kv, d_k, d_v, gated)")
    if R is not None and R.shape != (B, Tq, D):
        raise ValueError("residual must be (B, Tq, D)")
    kvl = _i32(kv_lengths)
    rws = _i32(rows)
    n_out = Tq if rws is None else len(rws)
    Y = np.empty((B, n_out, D), dtype=np.float64)
    fn = lib.oracle_mha_forward_rounded if round_bf16 else lib.oracle_mha_forward_ex
    rc = fn(B, Tq, Tkv, D, h, h_kv, d_k, d_v, int(bool(gated)), _ptr(Xq),
                                   _ptr(Xkv), _ptr(Wqkv), _ptr(bqkv), _ptr(Wo), _ptr(bo), _ptr(R),
                                   int(bool(causal)), _iptr(kvl), _iptr(rws),
                                   0 if rws is None else len(rws), _ptr(Y), nthreads)
    if rc:
        raise ValueError(f"oracle_mha_forward_ex failed ({rc})")
    return Y


def decode(Q, Kc, Vc, h: int, cache_lengths, h_kv=None, nthreads: int = 0):
    """One decode step: new query rows Q (B,Tq,h*dk) over the cache Kc (B,Tmax,h_kv*dk),
    Vc (B,Tmax,h_kv*dv); cache_lengths L_b count the cached tokens including the Tq new
    ones (the last Tq of them).  Returns O (B, Tq, h*dv)."""
    lib = _load()
    Q = _f64(Q)
    Kc = _f64(Kc)
    Vc = _f64(Vc)
    h_kv = h if h_kv is None else int(h_kv)
    B, Tq, hdk = Q.shape
    _, Tmax, kvw = Vc.shape
    if hdk % h or kvw % h_kv or h % h_kv:
        raise ValueError("head counts do not divide the widths")
    dk, dv = hdk // h, kvw // h_kv
    if Kc.shape != (B, Tmax, h_kv * dk):
        raise ValueError("K cache width is not h_kv * d_k")
    lens = _i32(cache_lengths)
    O = np.empty((B, Tq, h * dv), dtype=np.float64)
    rc = lib.oracle_decode(B, Tq, Tmax, h, h_kv, dk, dv, _ptr(Q), hdk, _ptr(Kc), h_kv * dk, _ptr(Vc),
                           kvw, _iptr(lens), _ptr(O), h * dv, nthreads)
    if rc:
        raise ValueError(f"oracle_decode failed ({rc})")
    return O
