"""Failure detection on the GPU without a fault: every pipeline wait in the kernels is
bounded.  mha_check_wait_timeout runs that same bounded wait on a barrier nothing ever
completes; the timeout must come back through the device status word, after about the
requested time, and the CUDA context must stay usable for a correct forward afterwards."""
import time

import numpy as np
import pytest

from gpu_util import assert_close, to_device, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_02_gb300 import Mha  # noqa: E402
from transformer_head_scaled_02_gb300 import _lib  # noqa: E402
from transformer_head_scaled_02_gb300 import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build_library()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def test_wait_timeout_is_reported_and_context_survives():
    w = wl.custom("after_timeout", B=2, T_q=200, D=256, h=4, d_k=64, causal=True)
    layer = Mha(w.D, w.h, w.d_k, dtype=torch.bfloat16)
    layer.ensure_workspace(w.B, w.T_q, w.T_kv)
    assert layer.status() == _lib.MHA_OK
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    _lib.mha_check_wait_timeout(layer.handle, 20_000_000, stream)   # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert layer.status() == _lib.MHA_ERR_TIMEOUT
    assert 0.019 <= dt < 5.0
    assert layer.status() == _lib.MHA_OK   # reading cleared it
    # the context is intact: a forward still runs and is correct
    x = wl.make_inputs(w, seed=9)
    d = {k: to_device(v, w.dtype) for k, v in x.items() if k != "kv_lengths"}
    y = layer.forward(d["X_q"], d["W_qkv"], d["b_qkv"], d["W_o"], d["b_o"], causal=True)
    torch.cuda.synchronize()
    assert layer.status() == _lib.MHA_OK
    ref = oracle.mha_forward(x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h, w.d_k,
                             w.d_v, causal=True)
    assert_close(to_host(y), ref, "bf16", "forward after a timed-out wait")
