"""ctypes binding of libmha.so (include/mha.h), one Python function per C entry
point with the same name and argument order.  Pointers are plain integers
(device addresses); streams are cudaStream_t handles as integers (0 = legacy
default stream).  Nothing here computes: every call goes to the library, and a
missing library is an ImportError -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmha.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "mha.h")

MHA_F32 = 0
MHA_BF16 = 1

MHA_OK = 0
MHA_ERR_INVALID_ARG = 1
MHA_ERR_UNSUPPORTED = 2
MHA_ERR_WORKSPACE = 3
MHA_ERR_CUDA = 4
MHA_ERR_TIMEOUT = 5
MHA_ERR_BAD_LENGTH = 6

_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

_SIGNATURES = {
    "mha_create": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _i]),
    "mha_create_ex": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _i, _i]),
    "mha_destroy": (None, [_vp]),
    "mha_workspace_size": (_sz, [_vp, _i, _i, _i]),
    "mha_set_workspace": (_i, [_vp, _vp, _sz]),
    "mha_forward": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp]),
    "mha_forward_checked": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp]),
    "mha_forward_ex": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp]),
    "mha_forward_host_workspace_size": (_sz, [_vp, _i, _i, _i, _i]),
    "mha_forward_host": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i,
                              _vp]),
    "mha_linear": (_i, [_vp, _vp, _i64, _i, _i, _vp, _i64, _i, _vp, _vp, _i64, _vp]),
    "mha_linear_ex": (_i, [_vp, _vp, _i64, _i, _i, _vp, _i64, _i, _vp, _vp, _i64, _vp, _i64, _vp]),
    "mha_linear_segments": (_i, [_vp, _vp, _i64, _i, _i, _vp, _i64, _i, _vp, _vp, _i, _vp, _i64, _vp]),
    "mha_linear_pair": (_i, [_vp, _vp, _i64, _i, _vp, _i64, _i, _vp, _vp, _i, _vp, _i64,
                             _vp, _i64, _i, _vp, _i64, _i, _vp, _vp, _i64, _i, _vp]),
    "mha_attention": (_i, [_vp, _i, _i, _i, _vp, _i64, _vp, _i64, _vp, _i64, _i, _vp, _vp, _i64,
                           _vp]),
    "mha_attention_ex": (_i, [_vp, _i, _i, _i, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i, _vp,
                              _vp, _i64, _vp]),
    "mha_decode_workspace_size": (_sz, [_vp, _i, _i, _i]),
    "mha_decode": (_i, [_vp, _i, _i, _i, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _vp]),
    "mha_get_status": (_i, [_vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "mha_forward_static_workspace": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp,
                                          _vp, _vp, _vp]),
    "mha_check_wait_timeout": (_i, [_vp, _i64, _vp]),
    "mha_strerror": (ctypes.c_char_p, [_i]),
}

_lib = None


class MhaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")


def header_symbols() -> list:
    """Names of the functions include/mha.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(mha_[a-z_]+)\s*\(", text)


def load():
    """Load libmha.so (raises ImportError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "(or python transformer_head_scaled_02_gb300/build.py)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(fn: str, code: int) -> int:
    if code != MHA_OK:
        raise MhaError(fn, code)
    return code


def strerror(code: int) -> str:
    return load().mha_strerror(int(code)).decode()


def mha_create(D: int, h: int, d_k: int, d_v: int, dtype: int) -> int:
    out = _vp()
    _check("mha_create", load().mha_create(ctypes.byref(out), D, h, d_k, d_v, dtype))
    return out.value


def mha_create_ex(D: int, h: int, h_kv: int, d_k: int, d_v: int, gated: int, dtype: int) -> int:
    out = _vp()
    _check("mha_create_ex", load().mha_create_ex(ctypes.byref(out), D, h, h_kv, d_k, d_v, int(gated),
                                                 dtype))
    return out.value


def mha_destroy(handle: int) -> None:
    load().mha_destroy(handle)


def mha_workspace_size(handle: int, B: int, T_q: int, T_kv: int) -> int:
    return int(load().mha_workspace_size(handle, B, T_q, T_kv))


def mha_set_workspace(handle: int, dev_ptr: int, nbytes: int) -> int:
    return _check("mha_set_workspace", load().mha_set_workspace(handle, dev_ptr, nbytes))


def mha_forward(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal, kv_lengths,
                out, stream, check: bool = True) -> int:
    code = load().mha_forward(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o,
                              int(causal), kv_lengths, out, stream)
    return _check("mha_forward", code) if check else code


def mha_forward_checked(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal,
                        kv_lengths, kv_lengths_host, out, stream, check: bool = True) -> int:
    """kv_lengths_host: a host int32 array (numpy) equal to the device kv_lengths, or None."""
    hp = None
    if kv_lengths_host is not None:
        import numpy as np
        arr = np.ascontiguousarray(kv_lengths_host, dtype=np.int32)
        hp = arr.ctypes.data_as(ctypes.c_void_p)
    code = load().mha_forward_checked(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o,
                                      int(causal), kv_lengths, hp, out, stream)
    return _check("mha_forward_checked", code) if check else code


def mha_forward_ex(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal, kv_lengths,
                   residual, out, stream, check: bool = True) -> int:
    code = load().mha_forward_ex(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o,
                                 int(causal), kv_lengths, residual, out, stream)
    return _check("mha_forward_ex", code) if check else code


def mha_forward_host_workspace_size(handle, B, T_q, T_kv, chunks) -> int:
    return load().mha_forward_host_workspace_size(handle, B, T_q, T_kv, chunks)


def mha_forward_host(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal, kv_lengths,
                     residual, out, chunks, stream, check: bool = True) -> int:
    code = load().mha_forward_host(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o,
                                   int(causal), kv_lengths, residual, out, chunks, stream)
    return _check("mha_forward_host", code) if check else code


def mha_linear(handle, A, lda, M, K, W, ldw, N, bias, C, ldc, stream, check: bool = True) -> int:
    code = load().mha_linear(handle, A, lda, M, K, W, ldw, N, bias, C, ldc, stream)
    return _check("mha_linear", code) if check else code


def mha_linear_ex(handle, A, lda, M, K, W, ldw, N, bias, R, ldr, C, ldc, stream,
                  check: bool = True) -> int:
    code = load().mha_linear_ex(handle, A, lda, M, K, W, ldw, N, bias, R, ldr, C, ldc, stream)
    return _check("mha_linear_ex", code) if check else code



def mha_linear_segments(handle, A, lda, M, K, W, ldw, N, bias, seg_len, seg_rows, C, ldc, stream,
                        check: bool = True):
    code = load().mha_linear_segments(handle, A, lda, M, K, W, ldw, N, bias, seg_len, seg_rows, C,
                                      ldc, stream)
    return _check("mha_linear_segments", code) if check else code

def mha_linear_pair(handle, A, lda, M, W, ldw, N, bias, seg_len, seg_rows, C, ldc, A2, lda2, M2, W2,
                    ldw2, N2, bias2, C2, ldc2, K, stream, check: bool = True):
    code = load().mha_linear_pair(handle, A, lda, M, W, ldw, N, bias, seg_len, seg_rows, C, ldc, A2,
                                  lda2, M2, W2, ldw2, N2, bias2, C2, ldc2, K, stream)
    return _check("mha_linear_pair", code) if check else code

def mha_attention(handle, B, T_q, T_kv, Q, ldq, K, ldk, V, ldv, causal, kv_lengths, O, ldo,
                  stream, check: bool = True) -> int:
    code = load().mha_attention(handle, B, T_q, T_kv, Q, ldq, K, ldk, V, ldv, int(causal),
                                kv_lengths, O, ldo, stream)
    return _check("mha_attention", code) if check else code


def mha_attention_ex(handle, B, T_q, T_kv, Q, ldq, K, ldk, V, ldv, G, ldg, causal, kv_lengths, O,
                     ldo, stream, check: bool = True) -> int:
    code = load().mha_attention_ex(handle, B, T_q, T_kv, Q, ldq, K, ldk, V, ldv, G, ldg, int(causal),
                                   kv_lengths, O, ldo, stream)
    return _check("mha_attention_ex", code) if check else code


def mha_decode_workspace_size(handle: int, B: int, T_q: int, T_max: int) -> int:
    return int(load().mha_decode_workspace_size(handle, B, T_q, T_max))


def mha_decode(handle, B, T_q, T_max, Q, ldq, K_cache, ldk, V_cache, ldv, cache_lengths, O, ldo,
               stream, check: bool = True) -> int:
    code = load().mha_decode(handle, B, T_q, T_max, Q, ldq, K_cache, ldk, V_cache, ldv,
                             cache_lengths, O, ldo, stream)
    return _check("mha_decode", code) if check else code


def mha_get_status(handle: int, stream: int) -> int:
    v = ctypes.c_int32(0)
    _check("mha_get_status", load().mha_get_status(handle, ctypes.byref(v), stream))
    return int(v.value)


def mha_check_wait_timeout(handle: int, limit_ns: int, stream, check: bool = True) -> int:
    """Run the kernels' bounded barrier wait against a barrier that never completes."""
    code = load().mha_check_wait_timeout(handle, limit_ns, stream)
    return _check("mha_check_wait_timeout", code) if check else code


MHA_STATIC_WORKSPACE_BYTES = 32 << 20


def mha_forward_static_workspace(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal,
                                 kv_lengths, out, status_out, stream, check: bool = True) -> int:
    """mha_forward with the library's own fixed scratch array instead of a caller workspace
    (for callers that may not allocate device memory; see include/mha.h).  status_out: device
    address of an int32 that receives the call's device status, or None."""
    code = load().mha_forward_static_workspace(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv,
                                               W_o, b_o, int(causal), kv_lengths, out, status_out,
                                               stream)
    return _check("mha_forward_static_workspace", code) if check else code
