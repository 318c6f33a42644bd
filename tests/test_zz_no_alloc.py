"""mha_forward_static_workspace: the forward for callers that may not allocate
device memory (a host framework that owns every allocation, or a serving loop
that cannot afford cudaMalloc's device-wide synchronisation).  Its scratch is a
fixed array inside the library instead of a caller workspace.

Called through the C ABI (ctypes), its output must match the ordinary
mha_forward (which uses a caller-attached workspace) within the parity
tolerances, on two calls in a row -- the second call runs on scratch that still
holds the first call's contents.  Sizes beyond the array are refused before
any CUDA work.  The file is named to be collected last and builds every input
itself, so it passes alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest

from gpu_util import assert_close, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

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


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_static_workspace_matches_mha_forward_twice(w):
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

        outs = []
        for _ in range(2):
            out = torch.full((w.B, w.T_q, w.D), float("nan"), dtype=torch_dtype(w.dtype),
                             device="cuda")
            _lib.mha_forward_static_workspace(handle, *ptrs, int(w.causal), _ptr(kvl),
                                              out.data_ptr(), stream)
            outs.append(out)
        torch.cuda.synchronize()
        assert _lib.mha_get_status(handle, stream) == _lib.MHA_OK
        r = to_host(ref)
        for out in outs:
            assert_close(to_host(out), r, w.dtype, f"{w.name} static workspace")
    finally:
        _lib.mha_destroy(handle)


def test_static_workspace_refuses_oversize():
    """A shape whose scratch exceeds the fixed array is refused before any
    CUDA work, and the output is left untouched."""
    w = wl.WORKLOADS["c3_bf16_causal"]  # 64 MiB of scratch > 32 MiB
    handle = _lib.mha_create(w.D, w.h, w.d_k, w.d_v, _lib.MHA_BF16)
    try:
        assert _lib.mha_workspace_size(handle, w.B, w.T_q, w.T_kv) > _lib.MHA_STATIC_WORKSPACE_BYTES
        out = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
        code = _lib.mha_forward_static_workspace(handle, 1 << 40, None, w.B, w.T_q, w.T_kv,
                                                 1 << 41, None, 1 << 42, None, 1, None,
                                                 out.data_ptr(), None, check=False)
        assert code == _lib.MHA_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert (out == 0).all()
    finally:
        _lib.mha_destroy(handle)
