"""The C-ABI library: it loads, exports every function include/mha.h declares,
and rejects bad arguments on the host before touching the GPU.  No test here
launches a kernel, so the file runs on a machine without a GPU."""
import ctypes

import pytest

from transformer_head_scaled_02_gb300 import _lib as L


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build_library()
    return L.load()


def test_exports_every_declared_symbol(lib):
    names = L.header_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_every_code(lib):
    for code in range(7):
        assert L.strerror(code) not in ("", "unknown status")
    assert L.strerror(99) == "unknown status"


def test_create_rejects_bad_sizes(lib):
    h = ctypes.c_void_p()
    for args in ((0, 8, 64, 64, 1), (512, 0, 64, 64, 1), (512, 8, -1, 64, 1),
                 (512, 8, 64, 0, 1), (512, 8, 64, 64, 7)):
        assert lib.mha_create(ctypes.byref(h), *args) == L.MHA_ERR_INVALID_ARG
    assert lib.mha_create(None, 512, 8, 64, 64, 1) == L.MHA_ERR_INVALID_ARG


def test_workspace_size_layout(lib):
    hdl = L.mha_create(1024, 16, 64, 64, L.MHA_BF16)
    try:
        # status 256 + Q (B*T*D*2) + KV (B*T*2D*2) + Ocat (B*T*D*2), each 256-aligned
        B, T, D = 4, 2048, 1024
        assert L.mha_workspace_size(hdl, B, T, T) == 256 + B * T * D * 2 * 4
        assert L.mha_workspace_size(hdl, -1, T, T) == 0
        assert L.mha_workspace_size(None, 1, 1, 1) == 0
    finally:
        L.mha_destroy(hdl)


def test_forward_rejects_bad_arguments_before_any_launch(lib):
    bf = L.mha_create(1024, 16, 64, 64, L.MHA_BF16)
    f32 = L.mha_create(64, 2, 32, 32, L.MHA_F32)
    odd = L.mha_create(96, 3, 32, 32, L.MHA_BF16)   # d_k = 32: no tensor-core kernel
    fake = 1 << 40                                   # never dereferenced: rejected earlier
    try:
        def fwd(h, **kw):
            a = dict(X_q=fake, X_kv=None, B=2, T_q=128, T_kv=128, W_qkv=fake, b_qkv=None,
                     W_o=fake, b_o=None, causal=0, kv_lengths=None, out=fake + (1 << 30),
                     stream=None)
            a.update(kw)
            return L.mha_forward(h, check=False, **a)
        assert fwd(None) == L.MHA_ERR_INVALID_ARG
        assert fwd(bf, B=-1) == L.MHA_ERR_INVALID_ARG
        assert fwd(bf, causal=1, X_kv=fake + (1 << 32), T_kv=256) == L.MHA_ERR_INVALID_ARG
        assert fwd(bf, T_kv=64) == L.MHA_ERR_INVALID_ARG          # self-attention needs T_kv == T_q
        assert fwd(bf, X_q=None) == L.MHA_ERR_INVALID_ARG
        assert fwd(bf, W_o=None) == L.MHA_ERR_INVALID_ARG
        assert fwd(bf, out=None) == L.MHA_ERR_INVALID_ARG
        assert fwd(bf, out=fake) == L.MHA_ERR_INVALID_ARG          # output aliases X_q
        assert fwd(bf, X_q=fake + 2) == L.MHA_ERR_INVALID_ARG      # bf16 needs 16-byte alignment
        assert fwd(bf) == L.MHA_ERR_WORKSPACE                       # no workspace attached
        assert fwd(odd) == L.MHA_ERR_UNSUPPORTED
        assert fwd(f32, X_q=fake + 4) == L.MHA_ERR_WORKSPACE        # fp32: no alignment rule
        assert fwd(bf, B=0) == L.MHA_OK                             # empty batch: nothing to do
        assert fwd(bf, T_q=0, T_kv=0) == L.MHA_OK
        assert fwd(bf, X_kv=fake + (1 << 32), T_kv=0) == L.MHA_ERR_INVALID_ARG
    finally:
        for h in (bf, f32, odd):
            L.mha_destroy(h)


def test_linear_and_attention_reject_bad_arguments(lib):
    bf = L.mha_create(1024, 16, 64, 64, L.MHA_BF16)
    fake = 1 << 40
    try:
        lin = lambda **kw: L.mha_linear(bf, **{**dict(A=fake, lda=64, M=10, K=64, W=fake + (1 << 30),
                                                      ldw=64, N=64, bias=None, C=fake + (1 << 32),
                                                      ldc=64, stream=None), **kw}, check=False)
        assert lin(K=0) == L.MHA_ERR_INVALID_ARG
        assert lin(K=60, lda=60) == L.MHA_ERR_INVALID_ARG           # bf16: K % 8
        assert lin(lda=32) == L.MHA_ERR_INVALID_ARG                 # lda < K
        assert lin(C=fake) == L.MHA_ERR_INVALID_ARG                 # C aliases A
        assert lin(M=0) == L.MHA_OK
        att = lambda **kw: L.mha_attention(bf, **{**dict(B=1, T_q=10, T_kv=10, Q=fake, ldq=3072,
                                                         K=fake + 2048, ldk=3072, V=fake + 4096,
                                                         ldv=3072, causal=0, kv_lengths=None,
                                                         O=fake + (1 << 32), ldo=1024,
                                                         stream=None), **kw}, check=False)
        assert att(ldq=1000) == L.MHA_ERR_INVALID_ARG               # < h*d_k
        assert att(causal=1, T_kv=11) == L.MHA_ERR_INVALID_ARG
        assert att(O=None) == L.MHA_ERR_INVALID_ARG
        assert att(T_q=0) == L.MHA_OK
    finally:
        L.mha_destroy(bf)


def test_wait_probe_rejects_bad_arguments(lib):
    hdl = L.mha_create(256, 4, 64, 64, L.MHA_BF16)
    try:
        assert L.mha_check_wait_timeout(None, 1000, None, check=False) == L.MHA_ERR_INVALID_ARG
        assert L.mha_check_wait_timeout(hdl, 0, None, check=False) == L.MHA_ERR_INVALID_ARG
        assert L.mha_check_wait_timeout(hdl, 20_000_000_000, None, check=False) == L.MHA_ERR_INVALID_ARG
        assert L.mha_check_wait_timeout(hdl, 1000, None, check=False) == L.MHA_ERR_WORKSPACE
    finally:
        L.mha_destroy(hdl)


def test_create_ex_validates_groups_and_gate(lib):
    h = ctypes.c_void_p()
    # h_kv must divide h and lie in [1, h]; gated is 0 or 1
    for args in ((512, 8, 3, 64, 64, 0, 1), (512, 8, 0, 64, 64, 0, 1), (512, 8, 16, 64, 64, 0, 1),
                 (512, 8, 8, 64, 64, 2, 1)):
        assert lib.mha_create_ex(ctypes.byref(h), *args) == L.MHA_ERR_INVALID_ARG
    for h_kv in (1, 2, 4, 8):
        hdl = L.mha_create_ex(512, 8, h_kv, 64, 64, 1, L.MHA_BF16)
        L.mha_destroy(hdl)


def test_workspace_size_grouped_and_gated(lib):
    # self-attention: status + [Q|G] region (B*T*(h*dk + h*dv)) + [K|V] (B*T*h_kv*(dk+dv)) + Ocat
    B, T, D, h, h_kv, d = 2, 256, 512, 8, 2, 64
    hdl = L.mha_create_ex(D, h, h_kv, d, d, 1, L.MHA_BF16)
    try:
        qg = B * T * (h * d + h * d) * 2
        kv = B * T * h_kv * 2 * d * 2
        oc = B * T * h * d * 2
        assert L.mha_workspace_size(hdl, B, T, T) == 256 + qg + kv + oc
    finally:
        L.mha_destroy(hdl)


def test_decode_and_linear_ex_reject_bad_arguments(lib):
    bf = L.mha_create_ex(1024, 16, 4, 64, 64, 0, L.MHA_BF16)
    odd = L.mha_create_ex(96, 3, 1, 32, 32, 0, L.MHA_BF16)   # d = 32: no tensor-core kernel
    fake = 1 << 40
    try:
        def dec(h, **kw):
            a = dict(B=2, T_q=1, T_max=1024, Q=fake, ldq=1024, K=fake, ldk=256, V=fake, ldv=256,
                     lens=fake, O=fake + (1 << 30), ldo=1024)
            a.update(kw)
            return L.mha_decode(h, a["B"], a["T_q"], a["T_max"], a["Q"], a["ldq"], a["K"], a["ldk"],
                                a["V"], a["ldv"], a["lens"], a["O"], a["ldo"], None, check=False)
        assert dec(None) == L.MHA_ERR_INVALID_ARG
        assert dec(bf, T_q=2000) == L.MHA_ERR_INVALID_ARG          # more new tokens than the cache
        assert dec(bf, lens=None) == L.MHA_ERR_INVALID_ARG
        assert dec(bf, ldk=128) == L.MHA_ERR_INVALID_ARG           # K row narrower than h_kv*d_k
        assert dec(bf, Q=fake + 2) == L.MHA_ERR_INVALID_ARG        # misaligned bf16 pointer
        assert dec(bf) == L.MHA_ERR_WORKSPACE                      # no workspace attached
        assert dec(odd, ldq=96, ldk=32, ldv=32, ldo=96) == L.MHA_ERR_UNSUPPORTED
        assert dec(bf, B=0) == L.MHA_OK and dec(bf, T_q=0) == L.MHA_OK
        assert L.mha_decode_workspace_size(bf, 2, 1, 1024) > 256
        assert L.mha_decode_workspace_size(None, 2, 1, 1024) == 0
        # status 256 + one (max, sum, d values) fp32 record per (batch, query head, new token,
        # split), splits at least two 128-key tiles long; 256-byte aligned
        for B, Tq, Tmax in ((2, 1, 1024), (32, 1, 8192), (3, 4, 300)):
            splits = (Tmax + 255) // 256
            part = 4 * B * 16 * Tq * splits * (64 + 2)
            assert L.mha_decode_workspace_size(bf, B, Tq, Tmax) == 256 + (part + 255) // 256 * 256
        assert L.mha_decode_workspace_size(bf, 0, 1, 1024) == 256
        assert L.mha_decode_workspace_size(bf, -1, 1, 1024) == 0

        def lin(**kw):
            a = dict(A=fake, lda=64, M=128, K=64, W=fake + (1 << 28), ldw=64, N=64, bias=None,
                     R=fake + (2 << 28), ldr=64, C=fake + (3 << 28), ldc=64)
            a.update(kw)
            return L.mha_linear_ex(bf, a["A"], a["lda"], a["M"], a["K"], a["W"], a["ldw"], a["N"],
                                   a["bias"], a["R"], a["ldr"], a["C"], a["ldc"], None, check=False)
        assert lin(ldr=32) == L.MHA_ERR_INVALID_ARG                 # residual row narrower than N
        assert lin(R=fake + (3 << 28) + 2) == L.MHA_ERR_INVALID_ARG # misaligned, overlapping C
        assert lin(R=fake + (3 << 28) + 64) == L.MHA_ERR_INVALID_ARG # partly overlaps C

        def seg(**kw):
            a = dict(A=fake, lda=64, M=512, K=64, W=fake + (1 << 28), ldw=64, N=64, bias=None,
                     lens=fake + (2 << 28), seg_rows=256, C=fake + (3 << 28), ldc=64)
            a.update(kw)
            return L.mha_linear_segments(bf, a["A"], a["lda"], a["M"], a["K"], a["W"], a["ldw"],
                                         a["N"], a["bias"], a["lens"], a["seg_rows"], a["C"], a["ldc"],
                                         None, check=False)
        assert seg(lens=None) == L.MHA_ERR_INVALID_ARG              # no segment lengths
        assert seg(seg_rows=0) == L.MHA_ERR_INVALID_ARG
        assert seg(seg_rows=300) == L.MHA_ERR_INVALID_ARG           # M not a multiple of it
        assert seg(ldc=32) == L.MHA_ERR_INVALID_ARG                 # as mha_linear: C row < N
        assert seg(A=fake + 2) == L.MHA_ERR_INVALID_ARG             # misaligned bf16 pointer
        assert seg(M=0) == L.MHA_OK

        def pair(**kw):
            a = dict(A=fake, lda=64, M=512, W=fake + (1 << 28), ldw=64, N=64, bias=None, lens=None,
                     seg_rows=0, C=fake + (3 << 28), ldc=64, A2=fake + (4 << 28), lda2=64, M2=300,
                     W2=fake + (5 << 28), ldw2=32, N2=32, bias2=None, C2=fake + (6 << 28), ldc2=32,
                     K=64)
            a.update(kw)
            return L.mha_linear_pair(bf, a["A"], a["lda"], a["M"], a["W"], a["ldw"], a["N"], a["bias"],
                                     a["lens"], a["seg_rows"], a["C"], a["ldc"], a["A2"], a["lda2"],
                                     a["M2"], a["W2"], a["ldw2"], a["N2"], a["bias2"], a["C2"],
                                     a["ldc2"], a["K"], None, check=False)
        assert pair(lens=fake + (7 << 28), seg_rows=0) == L.MHA_ERR_INVALID_ARG
        assert pair(lens=fake + (7 << 28), seg_rows=300) == L.MHA_ERR_INVALID_ARG  # M % 300
        assert pair(ldc2=16) == L.MHA_ERR_INVALID_ARG           # second output row < N2
        assert pair(A2=fake + (4 << 28) + 2) == L.MHA_ERR_INVALID_ARG  # misaligned bf16 pointer
        assert pair(C2=fake + (3 << 28) + 64) == L.MHA_ERR_INVALID_ARG  # outputs overlap
        assert pair(C2=fake + 128) == L.MHA_ERR_INVALID_ARG     # C2 over the first's A
        assert pair(C=fake + (5 << 28)) == L.MHA_ERR_INVALID_ARG  # C over the second's W
        assert pair(K=0) == L.MHA_ERR_INVALID_ARG
        assert pair(M=0, M2=0) == L.MHA_OK
    finally:
        L.mha_destroy(bf)
        L.mha_destroy(odd)


def test_forward_host_workspace_layout(lib):
    hdl = L.mha_create(1024, 16, 64, 64, L.MHA_BF16)
    try:
        B, T, D = 4, 2048, 1024
        act = B * T * D * 2
        # chunk scratch (for the largest chunk: 4; 2 + 2; 1 + 2 + 1; 1 each) + X_q, X_kv, residual,
        # Y copies
        for chunks, Bc in ((1, 4), (2, 2), (3, 2), (4, 1), (16, 1)):
            assert L.mha_forward_host_workspace_size(hdl, B, T, T, chunks) == \
                L.mha_workspace_size(hdl, Bc, T, T) + 4 * act
        assert L.mha_forward_host_workspace_size(hdl, B, T, T, 0) == 0
        assert L.mha_forward_host_workspace_size(hdl, B, T, T, 17) == 0
        assert L.mha_forward_host_workspace_size(hdl, 0, T, T, 1) == 0
        assert L.mha_forward_host_workspace_size(None, B, T, T, 1) == 0
    finally:
        L.mha_destroy(hdl)


def test_forward_checked_validates_host_lengths_before_any_launch(lib):
    import numpy as np
    hdl = L.mha_create(256, 4, 64, 64, L.MHA_BF16)
    fake = 1 << 40  # never dereferenced: every call below returns before any launch
    try:
        def fwd(lens_dev, lens_host, T_kv=100):
            return L.mha_forward_checked(hdl, fake, fake + (1 << 30), 3, 50, T_kv, fake + (2 << 30), None,
                                         fake + (3 << 30), None, 0, lens_dev, lens_host,
                                         fake + (4 << 30), None, check=False)
        good = np.array([1, 100, 37], dtype=np.int32)
        assert fwd(fake + (5 << 30), np.array([0, 100, 37], dtype=np.int32)) == L.MHA_ERR_BAD_LENGTH
        assert fwd(fake + (5 << 30), np.array([1, 101, 37], dtype=np.int32)) == L.MHA_ERR_BAD_LENGTH
        assert fwd(fake + (5 << 30), None) == L.MHA_ERR_INVALID_ARG   # device lengths, no host copy
        assert fwd(None, good) == L.MHA_ERR_INVALID_ARG                # host copy, no device lengths
        # valid lengths: on to mha_forward, which finds no workspace attached
        assert fwd(fake + (5 << 30), good) == L.MHA_ERR_WORKSPACE
        assert fwd(None, None) == L.MHA_ERR_WORKSPACE
    finally:
        L.mha_destroy(hdl)


def test_forward_host_rejects_bad_arguments_before_any_copy(lib):
    hdl = L.mha_create(1024, 16, 64, 64, L.MHA_BF16)
    fake = 1 << 40  # never dereferenced: every call below is rejected first
    try:
        def fwd(**kw):
            a = dict(X_q=fake, X_kv=None, B=2, T_q=128, T_kv=128, W_qkv=fake, b_qkv=None,
                     W_o=fake, b_o=None, causal=0, kv_lengths=None, residual=None,
                     out=fake + (1 << 30), chunks=2, stream=None)
            a.update(kw)
            return L.mha_forward_host(hdl, check=False, **a)
        assert L.mha_forward_host(None, fake, None, 2, 128, 128, fake, None, fake, None, 0, None,
                                  None, fake, 2, None, check=False) == L.MHA_ERR_INVALID_ARG
        assert fwd(chunks=0) == L.MHA_ERR_INVALID_ARG
        assert fwd(chunks=17) == L.MHA_ERR_INVALID_ARG
        assert fwd(T_kv=64) == L.MHA_ERR_INVALID_ARG           # self-attention needs T_kv == T_q
        assert fwd(out=fake) == L.MHA_ERR_INVALID_ARG          # out aliases X_q
        assert fwd(W_qkv=None) == L.MHA_ERR_INVALID_ARG
        assert fwd(B=0) == L.MHA_OK                            # empty batch: nothing to do
        assert fwd() == L.MHA_ERR_WORKSPACE                    # no workspace attached
    finally:
        L.mha_destroy(hdl)


def test_static_workspace_rejects_bad_arguments_before_any_cuda_call(lib):
    """mha_forward_static_workspace refuses every invalid call on the host, before it looks
    up or touches its scratch array (so these run without a GPU)."""
    bf = L.mha_create(1024, 16, 64, 64, L.MHA_BF16)
    fake = 1 << 40                                   # never dereferenced: rejected earlier
    try:
        def fwd(**kw):
            a = dict(X_q=fake, X_kv=None, B=1, T_q=128, T_kv=128, W_qkv=fake + (1 << 34),
                     b_qkv=None, W_o=fake + (1 << 35), b_o=None, causal=1, kv_lengths=None,
                     out=fake + (1 << 36), status_out=fake + (1 << 37), stream=None)
            a.update(kw)
            return L.mha_forward_static_workspace(bf, check=False, **a)
        assert L.mha_forward_static_workspace(None, fake, None, 1, 128, 128, fake, None, fake,
                                              None, 1, None, fake, None, None,
                                              check=False) == L.MHA_ERR_INVALID_ARG
        assert fwd(B=4, T_q=2048, T_kv=2048) == L.MHA_ERR_WORKSPACE  # 64 MiB > 32 MiB array
        assert fwd(X_q=fake + 2) == L.MHA_ERR_INVALID_ARG             # bf16 alignment
        assert fwd(out=fake) == L.MHA_ERR_INVALID_ARG                 # output aliases X_q
        assert fwd(T_kv=64) == L.MHA_ERR_INVALID_ARG                  # self-attention, T_kv != T_q
        assert fwd(status_out=fake + 2) == L.MHA_ERR_INVALID_ARG      # status word alignment
        assert fwd(B=0) == L.MHA_OK                                   # empty batch: nothing to do
    finally:
        L.mha_destroy(bf)
