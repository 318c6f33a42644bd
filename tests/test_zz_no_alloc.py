"""mha_forward_static_workspace: the forward for callers that may not allocate
device memory (a host framework that owns every allocation, or a serving loop
that cannot afford cudaMalloc's device-wide synchronisation).  Its scratch is a
fixed array inside the library instead of a caller workspace.

Called through the C ABI (ctypes), on two calls in a row -- the second runs on
scratch that still holds the first call's contents -- its output must match
both the fp64 oracle and the ordinary mha_forward (which uses a caller-attached
workspace) within the parity tolerances, its device status must read MHA_OK,
and the calls must leave the device's free memory unchanged.  A bad key length
on this path is reported through the caller's status word.  Sizes beyond the
array are refused before any CUDA work.  The file is named to be collected last
and builds every input itself, so it passes alone in a fresh process as well as
after the other tests.
"""
import numpy as np
import pytest

from gpu_util import assert_close, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_02_gb300 import _lib  # noqa: E402
from transformer_head_scaled_02_gb300 import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build_library()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _ptr(t):
    return None if t is None else t.data_ptr()


CASES = [
    wl.custom("static_bf16_causal", B=2, T_q=300, D=256, h=4, d_k=64, causal=True),
    wl.custom("static_bf16_cross", B=3, T_q=90, T_kv=260, D=256, h=2, d_k=128, cross=True,
              kv_len_range=(1, 260)),
    wl.WORKLOADS["c2_f32_causal"],
]


def _oracle(w, x):
    return oracle.mha_forward(x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h, w.d_k,
                              w.d_v, Xkv=x["X_kv"], causal=w.causal, kv_lengths=x["kv_lengths"])


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_static_workspace_matches_oracle_and_mha_forward_twice(w):
    x = wl.make_inputs(w, seed=11)
    d = {k: to_device(v, w.dtype) for k, v in x.items() if k != "kv_lengths"}
    kvl = None if x["kv_lengths"] is None else torch.from_numpy(x["kv_lengths"]).cuda()
    dt = _lib.MHA_BF16 if w.dtype == "bf16" else _lib.MHA_F32
    handle = _lib.mha_create(w.D, w.h, w.d_k, w.d_v, dt)
    stream = torch.cuda.current_stream().cuda_stream
    try:
        need = _lib.mha_workspace_size(handle, w.B, w.T_q, w.T_kv)
        assert 0 < need <= _lib.MHA_STATIC_WORKSPACE_BYTES
        args = (d["X_q"], d["X_kv"], w.B, w.T_q, w.T_kv, d["W_qkv"], d["b_qkv"], d["W_o"], d["b_o"])
        ptrs = [_ptr(a) if not isinstance(a, int) else a for a in args]

        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        _lib.mha_set_workspace(handle, ws.data_ptr(), need)
        ref = torch.empty((w.B, w.T_q, w.D), dtype=torch_dtype(w.dtype), device="cuda")
        _lib.mha_forward(handle, *ptrs, int(w.causal), _ptr(kvl), ref.data_ptr(), stream)

        outs = [torch.full((w.B, w.T_q, w.D), float("nan"), dtype=torch_dtype(w.dtype),
                           device="cuda") for _ in range(2)]
        status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        for i, out in enumerate(outs):
            if i == 1:
                free_before = torch.cuda.mem_get_info()[0]
            _lib.mha_forward_static_workspace(handle, *ptrs, int(w.causal), _ptr(kvl),
                                              out.data_ptr(), status[i:].data_ptr(), stream)
            torch.cuda.synchronize()
        # the second call allocated nothing on the device
        assert torch.cuda.mem_get_info()[0] == free_before
        # the static calls' device status, copied out to the caller's words
        assert status.tolist() == [_lib.MHA_OK, _lib.MHA_OK]
        # the handle's own workspace holds only the ordinary call's status
        assert _lib.mha_get_status(handle, stream) == _lib.MHA_OK
        r = to_host(ref)
        o = _oracle(w, x)
        assert_close(r, o, w.dtype, f"{w.name} mha_forward vs oracle")
        for out in outs:
            got = to_host(out)
            e = assert_close(got, o, w.dtype, f"{w.name} static workspace vs oracle")
            assert_close(got, r, w.dtype, f"{w.name} static workspace vs mha_forward")
            print(w.name, "static workspace vs oracle", e)
    finally:
        _lib.mha_destroy(handle)


def test_static_workspace_reports_bad_lengths_through_status_out():
    """Key lengths outside [1, T_kv] give NaN rows and MHA_ERR_BAD_LENGTH in the caller's
    status word; the next call, with valid lengths, starts from a clean status."""
    w = wl.custom("static_badlen", B=3, T_q=50, T_kv=140, D=128, h=2, d_k=64, cross=True,
                  kv_len_range=(1, 140))
    x = wl.make_inputs(w, seed=5)
    d = {k: to_device(v, w.dtype) for k, v in x.items() if k != "kv_lengths"}
    handle = _lib.mha_create(w.D, w.h, w.d_k, w.d_v, _lib.MHA_BF16)
    stream = torch.cuda.current_stream().cuda_stream
    try:
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        ptrs = [d["X_q"].data_ptr(), d["X_kv"].data_ptr(), w.B, w.T_q, w.T_kv,
                d["W_qkv"].data_ptr(), d["b_qkv"].data_ptr(), d["W_o"].data_ptr(),
                d["b_o"].data_ptr(), 0]
        bad = torch.tensor([0, 77, 141], dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.T_q, w.D), dtype=torch.bfloat16, device="cuda")
        _lib.mha_forward_static_workspace(handle, *ptrs, bad.data_ptr(), out.data_ptr(),
                                          status.data_ptr(), stream)
        torch.cuda.synchronize()
        assert int(status.item()) == _lib.MHA_ERR_BAD_LENGTH
        yh = to_host(out)
        assert np.isnan(yh[0]).all() and np.isnan(yh[2]).all()
        ref = _oracle(w, {**x, "kv_lengths": np.array([1, 77, 1], dtype=np.int32)})
        assert_close(yh[1], ref[1], "bf16", "valid batch next to invalid ones")
        good = torch.from_numpy(x["kv_lengths"]).cuda()
        _lib.mha_forward_static_workspace(handle, *ptrs, good.data_ptr(), out.data_ptr(),
                                          status.data_ptr(), stream)
        torch.cuda.synchronize()
        assert int(status.item()) == _lib.MHA_OK
        assert_close(to_host(out), _oracle(w, x), "bf16", "valid lengths after invalid ones")
    finally:
        _lib.mha_destroy(handle)


def test_static_workspace_refuses_before_touching_anything():
    """A shape whose scratch exceeds the fixed array, or any other invalid argument, is
    refused before any CUDA work: the output and the caller's status word stay as they were."""
    w = wl.WORKLOADS["c3_bf16_causal"]  # 64 MiB of scratch > 32 MiB
    handle = _lib.mha_create(w.D, w.h, w.d_k, w.d_v, _lib.MHA_BF16)
    try:
        assert _lib.mha_workspace_size(handle, w.B, w.T_q, w.T_kv) > _lib.MHA_STATIC_WORKSPACE_BYTES
        out = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
        status = torch.full((2,), 99, dtype=torch.int32, device="cuda")
        code = _lib.mha_forward_static_workspace(handle, 1 << 40, None, w.B, w.T_q, w.T_kv,
                                                 1 << 41, None, 1 << 42, None, 1, None,
                                                 out.data_ptr(), status.data_ptr(), None,
                                                 check=False)
        assert code == _lib.MHA_ERR_WORKSPACE
        # small enough, but X_q is not 16-byte aligned, or the status word not 4-byte aligned
        for xq, st in ((1 << 40 | 2, status.data_ptr()), (1 << 40, status.data_ptr() + 2)):
            code = _lib.mha_forward_static_workspace(handle, xq, None, 1, 128, 128, 1 << 41, None,
                                                     1 << 42, None, 1, None, out.data_ptr(), st,
                                                     None, check=False)
            assert code == _lib.MHA_ERR_INVALID_ARG
        torch.cuda.synchronize()
        assert (out == 0).all()
        assert status.tolist() == [99, 99]
    finally:
        _lib.mha_destroy(handle)
