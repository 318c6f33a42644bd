"""Torch-tensor front end of libmha.so.

torch supplies device memory and the current CUDA stream; every step of the
forward runs in the library's kernels.  This module only checks tensor
properties, allocates the caller-side buffers (output and workspace) and
passes raw pointers through the C ABI (see ``_lib``).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.MHA_F32, torch.bfloat16: _lib.MHA_BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


class Mha:
    """One multi-head attention layer shape: width D, h heads of d_k / d_v.

    ``forward`` computes MultiHead(X_q, X_kv) = Concat(head_1..head_h) W_o + b_o
    with head_i = softmax(Q_i K_i^T / sqrt(d_k) [+ mask]) V_i, the fused
    [Q|K|V] projection X W_qkv + b_qkv feeding it (itwiki.kr "멀티 헤드 어텐션",
    수식 and the tensor-shape table).  Variants (same page, 추론 비용과 변형):
    ``h_kv`` K/V heads shared by groups of query heads (MQA/GQA), ``gated`` sigmoid
    output gate (a fourth projection block [Q|K|V|G]); ``forward(residual=...)`` adds
    a residual in the output projection; ``decode`` attends new tokens to a KV cache.
    """

    def __init__(self, D: int, h: int, d_k: int, d_v: Optional[int] = None,
                 dtype: torch.dtype = torch.bfloat16, device=None, h_kv: Optional[int] = None,
                 gated: bool = False):
        if dtype not in _DTYPES:
            raise TypeError(f"dtype must be one of {list(_DTYPES)}")
        self.D, self.h, self.d_k = D, h, d_k
        self.d_v = d_k if d_v is None else d_v
        self.h_kv = h if h_kv is None else h_kv
        self.gated = bool(gated)
        self.dtype = dtype
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.handle = _lib.mha_create_ex(D, h, self.h_kv, d_k, self.d_v, int(self.gated),
                                         _DTYPES[dtype])
        self._ws: Optional[torch.Tensor] = None

    @property
    def proj_width(self) -> int:
        """Columns of the fused projection [Q | K | V (| G)]."""
        return (self.h * self.d_k + self.h_kv * (self.d_k + self.d_v)
                + (self.h * self.d_v if self.gated else 0))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            _lib.mha_destroy(h)
            self.handle = None

    # ------------------------------------------------------------ workspace
    def workspace_size(self, B: int, T_q: int, T_kv: int) -> int:
        return _lib.mha_workspace_size(self.handle, B, T_q, T_kv)

    def ensure_workspace(self, B: int, T_q: int, T_kv: int, need: Optional[int] = None) -> torch.Tensor:
        need = self.workspace_size(B, T_q, T_kv) if need is None else need
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
            _lib.mha_set_workspace(self.handle, self._ws.data_ptr(), self._ws.numel())
        return self._ws

    def status(self) -> int:
        """Read and clear the device status word (synchronises the current stream)."""
        return _lib.mha_get_status(self.handle, _stream())

    # ------------------------------------------------------------ checks
    def _check(self, name, t, shape=None):
        if t is None:
            return
        if not t.is_cuda or t.dtype != self.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {self.dtype} CUDA tensor")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")

    # ------------------------------------------------------------ the layer
    def forward(self, X_q: torch.Tensor, W_qkv: torch.Tensor, b_qkv: Optional[torch.Tensor],
                W_o: torch.Tensor, b_o: Optional[torch.Tensor], X_kv: Optional[torch.Tensor] = None,
                causal: bool = False, kv_lengths: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None,
                residual: Optional[torch.Tensor] = None) -> torch.Tensor:
        B, T_q, D = X_q.shape
        T_kv = T_q if X_kv is None else X_kv.shape[1]
        ncols = self.proj_width
        self._check("X_q", X_q, (B, T_q, self.D))
        self._check("X_kv", X_kv, None if X_kv is None else (B, T_kv, self.D))
        self._check("W_qkv", W_qkv, (self.D, ncols))
        self._check("b_qkv", b_qkv, None if b_qkv is None else (ncols,))
        self._check("W_o", W_o, (self.h * self.d_v, self.D))
        self._check("b_o", b_o, None if b_o is None else (self.D,))
        if kv_lengths is not None and (kv_lengths.dtype != torch.int32 or not kv_lengths.is_cuda
                                       or kv_lengths.numel() != B):
            raise ValueError("kv_lengths must be a CUDA int32 tensor of length B")
        if out is None:
            out = torch.empty((B, T_q, self.D), dtype=self.dtype, device=X_q.device)
        self._check("out", out, (B, T_q, self.D))
        self._check("residual", residual, None if residual is None else (B, T_q, self.D))
        self.ensure_workspace(B, T_q, T_kv)
        _lib.mha_forward_ex(self.handle, _ptr(X_q), _ptr(X_kv), B, T_q, T_kv, _ptr(W_qkv),
                            _ptr(b_qkv), _ptr(W_o), _ptr(b_o), causal, _ptr(kv_lengths),
                            _ptr(residual), _ptr(out), _stream())
        return out

    __call__ = forward

    def forward_host(self, X_q: torch.Tensor, W_qkv: torch.Tensor, b_qkv: Optional[torch.Tensor],
                     W_o: torch.Tensor, b_o: Optional[torch.Tensor], out: torch.Tensor,
                     X_kv: Optional[torch.Tensor] = None, causal: bool = False,
                     kv_lengths: Optional[torch.Tensor] = None,
                     residual: Optional[torch.Tensor] = None, chunks: int = 4) -> torch.Tensor:
        """forward() with X_q, X_kv, residual and out in (pinned) host memory and the weights on
        the device: the batch goes through in chunks whose copies overlap the kernels.  Enqueued
        on the current stream; synchronise it before reading ``out``."""
        B, T_q, D = X_q.shape
        T_kv = T_q if X_kv is None else X_kv.shape[1]
        for name, t, T in (("X_q", X_q, T_q), ("X_kv", X_kv, T_kv), ("residual", residual, T_q),
                           ("out", out, T_q)):
            if t is None:
                continue
            if t.is_cuda or t.dtype != self.dtype or not t.is_contiguous() or tuple(t.shape) != (B, T, self.D):
                raise ValueError(f"{name} must be a contiguous host {self.dtype} tensor of shape "
                                 f"{(B, T, self.D)}")
        self._check("W_qkv", W_qkv, (self.D, self.proj_width))
        self._check("b_qkv", b_qkv, None if b_qkv is None else (self.proj_width,))
        self._check("W_o", W_o, (self.h * self.d_v, self.D))
        self._check("b_o", b_o, None if b_o is None else (self.D,))
        if kv_lengths is not None and (kv_lengths.dtype != torch.int32 or not kv_lengths.is_cuda
                                       or kv_lengths.numel() != B):
            raise ValueError("kv_lengths must be a CUDA int32 tensor of length B")
        need = _lib.mha_forward_host_workspace_size(self.handle, B, T_q, T_kv, chunks)
        if need == 0:
            raise ValueError("invalid size or chunk count")
        self.ensure_workspace(B, T_q, T_kv, need=need)
        _lib.mha_forward_host(self.handle, _ptr(X_q), _ptr(X_kv), B, T_q, T_kv, _ptr(W_qkv),
                              _ptr(b_qkv), _ptr(W_o), _ptr(b_o), causal, _ptr(kv_lengths),
                              _ptr(residual), _ptr(out), chunks, _stream())
        return out

    # ------------------------------------------------------------ single steps
    def linear(self, A: torch.Tensor, W: torch.Tensor, bias: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None,
               residual: Optional[torch.Tensor] = None) -> torch.Tensor:
        """C = A W + bias (+ residual) for 2-D A (M, K), W (K, N), residual (M, N) (row strides
        may exceed the width)."""
        M, K = A.shape
        N = W.shape[1]
        if out is None:
            out = torch.empty((M, N), dtype=self.dtype, device=A.device)
        mats = [("A", A), ("W", W), ("out", out)] + ([("residual", residual)] if residual is not None else [])
        for name, t in mats:
            if not t.is_cuda or t.dtype != self.dtype or t.stride(1) != 1:
                raise ValueError(f"{name} must be a row-major {self.dtype} CUDA matrix")
        self._check("bias", bias, None if bias is None else (N,))
        _lib.mha_linear_ex(self.handle, _ptr(A), A.stride(0), M, K, _ptr(W), W.stride(0), N,
                           _ptr(bias), _ptr(residual), 0 if residual is None else residual.stride(0),
                           _ptr(out), out.stride(0), _stream())
        return out

    def linear_segments(self, A: torch.Tensor, W: torch.Tensor, bias: Optional[torch.Tensor],
                        seg_len: torch.Tensor, seg_rows: int,
                        out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """C = A W + bias where only the rows that whole 128-row tiles up to each segment's
        length need are guaranteed: the key/value projection of cross-attention with key
        lengths seg_len (CUDA int32, one per segment of seg_rows rows)."""
        M, K = A.shape
        N = W.shape[1]
        if out is None:
            out = torch.empty((M, N), dtype=self.dtype, device=A.device)
        for name, t in (("A", A), ("W", W), ("out", out)):
            if not t.is_cuda or t.dtype != self.dtype or t.stride(1) != 1:
                raise ValueError(f"{name} must be a row-major {self.dtype} CUDA matrix")
        self._check("bias", bias, None if bias is None else (N,))
        if seg_len.dtype != torch.int32 or not seg_len.is_cuda:
            raise ValueError("seg_len must be a CUDA int32 tensor")
        _lib.mha_linear_segments(self.handle, _ptr(A), A.stride(0), M, K, _ptr(W), W.stride(0), N,
                                 _ptr(bias), _ptr(seg_len), seg_rows, _ptr(out), out.stride(0),
                                 _stream())
        return out

    def linear_pair(self, A: torch.Tensor, W: torch.Tensor, bias: Optional[torch.Tensor],
                    A2: torch.Tensor, W2: torch.Tensor, bias2: Optional[torch.Tensor],
                    seg_len: Optional[torch.Tensor] = None, seg_rows: int = 0,
                    out: Optional[torch.Tensor] = None,
                    out2: Optional[torch.Tensor] = None):
        """(A W + bias, A2 W2 + bias2) in one launch where possible (the cross-attention key /
        value and query projections); with seg_len, rows of the first past each segment's
        length may be left unwritten as in linear_segments.  Returns (out, out2)."""
        M, K = A.shape
        M2, K2 = A2.shape
        N, N2 = W.shape[1], W2.shape[1]
        if K2 != K or W.shape[0] != K or W2.shape[0] != K:
            raise ValueError("both projections need the same inner dimension")
        if out is None:
            out = torch.empty((M, N), dtype=self.dtype, device=A.device)
        if out2 is None:
            out2 = torch.empty((M2, N2), dtype=self.dtype, device=A.device)
        for name, t in (("A", A), ("W", W), ("out", out), ("A2", A2), ("W2", W2), ("out2", out2)):
            if not t.is_cuda or t.dtype != self.dtype or t.stride(1) != 1:
                raise ValueError(f"{name} must be a row-major {self.dtype} CUDA matrix")
        self._check("bias", bias, None if bias is None else (N,))
        self._check("bias2", bias2, None if bias2 is None else (N2,))
        if seg_len is not None and (seg_len.dtype != torch.int32 or not seg_len.is_cuda):
            raise ValueError("seg_len must be a CUDA int32 tensor")
        _lib.mha_linear_pair(self.handle, _ptr(A), A.stride(0), M, _ptr(W), W.stride(0), N, _ptr(bias),
                             _ptr(seg_len), seg_rows, _ptr(out), out.stride(0), _ptr(A2), A2.stride(0),
                             M2, _ptr(W2), W2.stride(0), N2, _ptr(bias2), _ptr(out2), out2.stride(0), K,
                             _stream())
        return out, out2

    def attention(self, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, causal: bool = False,
                  kv_lengths: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None,
                  G: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Attention of all heads over (B, T, width) views whose last dim is contiguous;
        head i uses columns [i*d, (i+1)*d) of Q (and of the gate pre-activations G), K/V
        head i // (h // h_kv).  Returns Ocat (B, T_q, h*d_v)."""
        B, T_q, _ = Q.shape
        T_kv = K.shape[1]
        views = [("Q", Q), ("K", K), ("V", V)] + ([("G", G)] if G is not None else [])
        for name, t in views:
            if not t.is_cuda or t.dtype != self.dtype or t.stride(2) != 1 \
                    or t.stride(0) != t.shape[1] * t.stride(1):
                raise ValueError(f"{name} must be a (B,T,*) {self.dtype} CUDA view with "
                                 "contiguous rows and batches")
        if out is None:
            out = torch.empty((B, T_q, self.h * self.d_v), dtype=self.dtype, device=Q.device)
        if kv_lengths is not None and (kv_lengths.dtype != torch.int32 or not kv_lengths.is_cuda):
            raise ValueError("kv_lengths must be a CUDA int32 tensor")
        _lib.mha_attention_ex(self.handle, B, T_q, T_kv, _ptr(Q), Q.stride(1), _ptr(K), K.stride(1),
                              _ptr(V), V.stride(1), _ptr(G), 0 if G is None else G.stride(1), causal,
                              _ptr(kv_lengths), _ptr(out), out.stride(1), _stream())
        return out

    def decode(self, Q: torch.Tensor, K_cache: torch.Tensor, V_cache: torch.Tensor,
               cache_lengths: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """One decode step: the T_q new tokens' queries Q (B, T_q, h*d_k view) over the cache
        K_cache (B, T_max, h_kv*d_k view), V_cache (B, T_max, h_kv*d_v view); cache_lengths
        (int32, B) count the cached tokens including the new ones.  Returns (B, T_q, h*d_v)."""
        B, T_q, _ = Q.shape
        T_max = K_cache.shape[1]
        for name, t in (("Q", Q), ("K_cache", K_cache), ("V_cache", V_cache)):
            if not t.is_cuda or t.dtype != self.dtype or t.stride(2) != 1 \
                    or t.stride(0) != t.shape[1] * t.stride(1):
                raise ValueError(f"{name} must be a (B,T,*) {self.dtype} CUDA view with "
                                 "contiguous rows and batches")
        if cache_lengths.dtype != torch.int32 or not cache_lengths.is_cuda or cache_lengths.numel() != B:
            raise ValueError("cache_lengths must be a CUDA int32 tensor of length B")
        if out is None:
            out = torch.empty((B, T_q, self.h * self.d_v), dtype=self.dtype, device=Q.device)
        self.ensure_workspace(B, T_q, T_max,
                              need=_lib.mha_decode_workspace_size(self.handle, B, T_q, T_max))
        _lib.mha_decode(self.handle, B, T_q, T_max, _ptr(Q), Q.stride(1), _ptr(K_cache),
                        K_cache.stride(1), _ptr(V_cache), V_cache.stride(1), _ptr(cache_lengths),
                        _ptr(out), out.stride(1), _stream())
        return out
