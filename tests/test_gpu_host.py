"""GPU tests of mha_forward_host, the forward with its activations in host memory: the batch
goes through in chunks of whole batch elements whose copies overlap the kernels.  Every batch
element is an independent problem (itwiki.kr "멀티 헤드 어텐션", tensor-shape table: the batch
axis is carried through every step), so the result must equal the device forward over the
whole batch bit for bit, and the fp64 oracle within the tolerances of tests/gpu_util.py.
"""
import math

import numpy as np
import pytest

from gpu_util import assert_close, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_02_gb300 import Mha  # noqa: E402
from transformer_head_scaled_02_gb300 import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _pinned(t):
    return t.cpu().pin_memory()


def _case(seed, dtype, B, Tq, D, h, d, Tkv=None, cross=False, lengths=None):
    Tkv = Tq if Tkv is None else Tkv
    width = oracle.proj_width(h, d, d, h, False)
    return {
        "X_q": wl.random_tensor((B, Tq, D), seed, dtype),
        "X_kv": wl.random_tensor((B, Tkv, D), seed + 1, dtype) if cross else None,
        "W_qkv": wl.random_tensor((D, width), seed + 2, dtype, scale=1.0 / math.sqrt(D)),
        "b_qkv": wl.random_tensor((width,), seed + 3, dtype, scale=0.1),
        "W_o": wl.random_tensor((h * d, D), seed + 4, dtype, scale=1.0 / math.sqrt(h * d)),
        "b_o": wl.random_tensor((D,), seed + 5, dtype, scale=0.1),
        "R": wl.random_tensor((B, Tq, D), seed + 6, dtype),
        "kv_lengths": None if lengths is None else np.asarray(lengths, dtype=np.int32),
    }


def _run(x, dtype, D, h, d, causal, residual, chunks):
    """(host-path output, device-path output) on the same layer and inputs."""
    layer = Mha(D, h, d, d, dtype=torch_dtype(dtype))
    t = {k: to_device(v, dtype) for k, v in x.items() if k != "kv_lengths"}
    kvl = None if x["kv_lengths"] is None else torch.from_numpy(x["kv_lengths"]).cuda()
    R = None
    if residual == "separate":
        R = t["R"]
    elif residual == "x":
        R = t["X_q"]
    ref_dev = layer.forward(t["X_q"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], X_kv=t["X_kv"],
                            causal=causal, kv_lengths=kvl, residual=R)
    xh = _pinned(t["X_q"])
    xkvh = None if t["X_kv"] is None else _pinned(t["X_kv"])
    rh = None if R is None else (xh if residual == "x" else _pinned(R))
    yh = torch.empty(ref_dev.shape, dtype=ref_dev.dtype).pin_memory()
    yh.fill_(float("nan"))
    layer.forward_host(xh, t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], out=yh, X_kv=xkvh,
                       causal=causal, kv_lengths=kvl, residual=rh, chunks=chunks)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return yh, ref_dev.cpu()


def _oracle(x, h, d, causal, residual):
    R = {"separate": x["R"], "x": x["X_q"], None: None}[residual]
    return oracle.mha_forward(x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], h, d, d,
                              Xkv=x["X_kv"], causal=causal, kv_lengths=x["kv_lengths"],
                              residual=R)


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 32)])
@pytest.mark.parametrize("chunks", [1, 2, 3, 16])
def test_host_forward_self_causal(dtype, d, chunks):
    h = 4
    D = h * d
    B, T = 5, 200 if dtype == "bf16" else 40   # 5 batch elements: chunks of 3+2, 1+3+1, 1 each
    x = _case(90, dtype, B, T, D, h, d)
    got, dev = _run(x, dtype, D, h, d, True, None, chunks)
    assert torch.equal(got.view(torch.int16 if dtype == "bf16" else torch.int32),
                       dev.view(torch.int16 if dtype == "bf16" else torch.int32))
    assert_close(to_host(got), _oracle(x, h, d, True, None), dtype, f"host forward chunks={chunks}")


@pytest.mark.parametrize("residual", ["separate", "x"])
def test_host_forward_cross_lengths_residual(residual):
    h, d = 4, 64
    D = h * d
    B, Tq, Tkv = 3, 130, 300
    x = _case(91, "bf16", B, Tq, D, h, d, Tkv=Tkv, cross=True, lengths=[Tkv, 17, Tkv - 40])
    got, dev = _run(x, "bf16", D, h, d, False, residual, 2)
    assert torch.equal(got.view(torch.int16), dev.view(torch.int16))
    assert_close(to_host(got), _oracle(x, h, d, False, residual), "bf16", f"host cross {residual}")


def test_host_forward_d128_repeated_calls():
    """Two calls back to back on one stream reuse the handle's copy buffers safely."""
    h, d = 2, 128
    D = h * d
    B, T = 4, 256
    x1 = _case(92, "bf16", B, T, D, h, d)
    x2 = _case(93, "bf16", B, T, D, h, d)
    layer = Mha(D, h, d, d, dtype=torch.bfloat16)
    outs, keep = [], []  # host inputs stay alive until the stream has read them
    for x in (x1, x2):
        t = {k: to_device(v, "bf16") for k, v in x.items() if k != "kv_lengths"}
        xh = _pinned(t["X_q"])
        yh = torch.empty((B, T, D), dtype=torch.bfloat16).pin_memory()
        layer.forward_host(xh, t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], out=yh, causal=True,
                           chunks=4)
        outs.append(yh)
        keep.append((xh, t))
    torch.cuda.synchronize()
    assert layer.status() == 0
    for x, yh in zip((x1, x2), outs):
        assert_close(to_host(yh), _oracle(x, h, d, True, None), "bf16", "host d128 repeated")
