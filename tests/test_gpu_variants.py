"""GPU parity of the variants (itwiki.kr "멀티 헤드 어텐션", section 추론 비용과 변형;
iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", sections 14 and 16): grouped K/V
heads (MQA/GQA), the sigmoid output gate, the fused residual, and the KV-cache decode step,
each against the fp64 oracle on the same seeded (bf16-rounded) inputs, through the C ABI.
Shapes span several tiles with ragged tails; the tolerances are those of tests/gpu_util.py.
"""
import math

import numpy as np
import pytest

from gpu_util import assert_close, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_02_gb300 import Mha  # noqa: E402
from transformer_head_scaled_02_gb300 import _lib  # noqa: E402
from transformer_head_scaled_02_gb300 import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _inputs(seed, dtype, B, Tq, D, h, d, h_kv, gated, Tkv=None, cross=False, lengths=None):
    """Seeded layer inputs: X ~ N(0,1), W ~ N(0, 1/D) (bf16-rounded for bf16)."""
    Tkv = Tq if Tkv is None else Tkv
    width = oracle.proj_width(h, d, d, h_kv, gated)
    x = {
        "X_q": wl.random_tensor((B, Tq, D), seed, dtype),
        "X_kv": wl.random_tensor((B, Tkv, D), seed + 1, dtype) if cross else None,
        "W_qkv": wl.random_tensor((D, width), seed + 2, dtype, scale=1.0 / math.sqrt(D)),
        "b_qkv": wl.random_tensor((width,), seed + 3, dtype, scale=0.1),
        "W_o": wl.random_tensor((h * d, D), seed + 4, dtype, scale=1.0 / math.sqrt(h * d)),
        "b_o": wl.random_tensor((D,), seed + 5, dtype, scale=0.1),
        "R": wl.random_tensor((B, Tq, D), seed + 6, dtype),
        "kv_lengths": None if lengths is None else np.asarray(lengths, dtype=np.int32),
    }
    return x


def _gpu_forward(x, dtype, D, h, d, h_kv, gated, causal, residual, Tkv=None):
    layer = Mha(D, h, d, d, dtype=torch_dtype(dtype), h_kv=h_kv, gated=gated)
    t = {k: to_device(v, dtype) for k, v in x.items() if k != "kv_lengths"}
    kvl = None if x["kv_lengths"] is None else torch.from_numpy(x["kv_lengths"]).cuda()
    y = layer.forward(t["X_q"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], X_kv=t["X_kv"],
                      causal=causal, kv_lengths=kvl, residual=t["R"] if residual else None)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return to_host(y)


def _oracle_forward(x, h, d, h_kv, gated, causal, residual):
    return oracle.mha_forward(x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], h, d, d,
                              Xkv=x["X_kv"], causal=causal, kv_lengths=x["kv_lengths"], h_kv=h_kv,
                              gated=gated, residual=x["R"] if residual else None)


# ------------------------------------------------------------------ grouped K/V heads

@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 32)])
@pytest.mark.parametrize("h_kv", [1, 2])
@pytest.mark.parametrize("causal", [True, False])
def test_grouped_heads_self_attention(dtype, d, h_kv, causal):
    h = 4
    D = h * d
    B, T = 2, 300 if dtype == "bf16" else 70
    x = _inputs(10 + h_kv, dtype, B, T, D, h, d, h_kv, False)
    got = _gpu_forward(x, dtype, D, h, d, h_kv, False, causal, False)
    ref = _oracle_forward(x, h, d, h_kv, False, causal, False)
    assert_close(got, ref, dtype, f"GQA h_kv={h_kv} d={d} causal={causal}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 32)])
def test_grouped_heads_cross_attention_with_key_lengths(dtype, d):
    h, h_kv = 8, 2
    D = h * d
    B, Tq, Tkv = 3, 130, 400 if dtype == "bf16" else 90
    lengths = [Tkv, 1, Tkv // 2 + 3]
    x = _inputs(20, dtype, B, Tq, D, h, d, h_kv, False, Tkv=Tkv, cross=True, lengths=lengths)
    got = _gpu_forward(x, dtype, D, h, d, h_kv, False, False, False, Tkv=Tkv)
    ref = _oracle_forward(x, h, d, h_kv, False, False, False)
    assert_close(got, ref, dtype, "GQA cross")


# ------------------------------------------------------------------ output gate

@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 32)])
@pytest.mark.parametrize("causal", [True, False])
def test_gated_self_attention(dtype, d, causal):
    h = 4
    D = h * d
    B, T = 2, 260 if dtype == "bf16" else 50
    x = _inputs(30, dtype, B, T, D, h, d, h, True)
    got = _gpu_forward(x, dtype, D, h, d, h, True, causal, False)
    ref = _oracle_forward(x, h, d, h, True, causal, False)
    assert_close(got, ref, dtype, f"gated d={d} causal={causal}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 32)])
def test_gated_cross_attention(dtype, d):
    h = 4
    D = h * d
    B, Tq, Tkv = 2, 140, 300 if dtype == "bf16" else 60
    x = _inputs(31, dtype, B, Tq, D, h, d, h, True, Tkv=Tkv, cross=True, lengths=[Tkv, Tkv - 7])
    got = _gpu_forward(x, dtype, D, h, d, h, True, False, False, Tkv=Tkv)
    ref = _oracle_forward(x, h, d, h, True, False, False)
    assert_close(got, ref, dtype, "gated cross")


# ------------------------------------------------------------------ residual

@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 32)])
def test_residual_forward(dtype, d):
    h = 4
    D = h * d
    B, T = 2, 200 if dtype == "bf16" else 40
    x = _inputs(40, dtype, B, T, D, h, d, h, False)
    got = _gpu_forward(x, dtype, D, h, d, h, False, True, True)
    ref = _oracle_forward(x, h, d, h, False, True, True)
    assert_close(got, ref, dtype, f"residual d={d}")


@pytest.mark.parametrize("B,T,d,h_kv,gated,causal", [
    (1, 100, 64, 4, False, True),    # 100 rows: both projections split K over clusters
    (2, 64, 128, 2, True, False),    # 128 rows, grouped heads and the gate
    (3, 5, 64, 1, False, True),      # 15 rows (a decode-sized batch), one K/V head
])
def test_few_row_forward_with_residual(B, T, d, h_kv, gated, causal):
    """Forwards of at most 128 rows: the projections (the output one with the residual in its
    epilogue) take the few-row split kernel; the whole layer equals the oracle's."""
    h = 4
    D = h * d
    x = _inputs(70, "bf16", B, T, D, h, d, h_kv, gated)
    got = _gpu_forward(x, "bf16", D, h, d, h_kv, gated, causal, True)
    ref = _oracle_forward(x, h, d, h_kv, gated, causal, True)
    assert_close(got, ref, "bf16", f"few-row forward B={B} T={T} d={d}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_residual_in_place_and_as_input(dtype):
    """residual == out (in place) and residual == X_q (the pages' X' = X + O W_O)."""
    h, d = 4, 64 if dtype == "bf16" else 32
    D = h * d
    B, T = 2, 150 if dtype == "bf16" else 40
    x = _inputs(41, dtype, B, T, D, h, d, h, False)
    layer = Mha(D, h, d, d, dtype=torch_dtype(dtype))
    t = {k: to_device(v, dtype) for k, v in x.items() if k != "kv_lengths"}
    out = t["R"].clone()
    layer.forward(t["X_q"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], causal=True, out=out,
                  residual=out)
    y2 = layer.forward(t["X_q"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], causal=True,
                       residual=t["X_q"])
    torch.cuda.synchronize()
    ref = _oracle_forward(x, h, d, h, False, True, True)
    assert_close(to_host(out), ref, dtype, "residual in place")
    x2 = dict(x)
    x2["R"] = x["X_q"]
    ref2 = _oracle_forward(x2, h, d, h, False, True, True)
    assert_close(to_host(y2), ref2, dtype, "residual = X_q")


# ------------------------------------------------------------------ all variants together

@pytest.mark.parametrize("d", [64, 128])
def test_grouped_gated_residual_forward(d):
    h, h_kv = 8, 2
    D = h * d
    B, T = 2, 384
    x = _inputs(50, "bf16", B, T, D, h, d, h_kv, True)
    got = _gpu_forward(x, "bf16", D, h, d, h_kv, True, True, True)
    ref = _oracle_forward(x, h, d, h_kv, True, True, True)
    assert_close(got, ref, "bf16", f"GQA+gate+residual d={d}")


# ------------------------------------------------------------------ decode

def _decode_case(seed, dtype, B, Tq, Tmax, h, h_kv, d, lengths):
    Q = wl.random_tensor((B, Tq, h * d), seed, dtype)
    Kc = wl.random_tensor((B, Tmax, h_kv * d), seed + 1, dtype)
    Vc = wl.random_tensor((B, Tmax, h_kv * d), seed + 2, dtype)
    layer = Mha(h * d, h, d, d, dtype=torch_dtype(dtype), h_kv=h_kv)
    lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    O = layer.decode(to_device(Q, dtype), to_device(Kc, dtype), to_device(Vc, dtype), lens)
    torch.cuda.synchronize()
    ref = oracle.decode(Q, Kc, Vc, h, lengths, h_kv=h_kv)
    return layer, to_host(O), ref


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 32)])
@pytest.mark.parametrize("h_kv", [8, 2, 1])
@pytest.mark.parametrize("Tq", [1, 4])
def test_decode_step(dtype, d, h_kv, Tq):
    h = 8
    B, Tmax = 3, 1000 if dtype == "bf16" else 200
    lengths = [Tmax, Tq + 5, Tmax // 2 + 77]
    layer, got, ref = _decode_case(60 + h_kv + Tq, dtype, B, Tq, Tmax, h, h_kv, d, lengths)
    assert layer.status() == 0
    assert_close(got, ref, dtype, f"decode h_kv={h_kv} Tq={Tq} d={d}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 32)])
def test_decode_invalid_lengths(dtype, d):
    h, h_kv, Tq, Tmax = 4, 2, 2, 300
    lengths = [Tmax, 1, Tmax + 1]  # valid, shorter than the new tokens, beyond the cache
    layer, got, ref = _decode_case(70, dtype, 3, Tq, Tmax, h, h_kv, d, lengths)
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()
    assert_close(got[0], ref[0], dtype, "decode valid batch beside invalid ones")
    assert layer.status() == _lib.MHA_ERR_BAD_LENGTH
    assert layer.status() == 0  # reading clears it


def test_decode_long_cache_many_groups():
    """Cache length not a multiple of the split, MQA over 16 heads, one new token."""
    h, h_kv, d, Tq = 16, 1, 64, 1
    B, Tmax = 2, 4133
    layer, got, ref = _decode_case(80, "bf16", B, Tq, Tmax, h, h_kv, d, [Tmax, 2049])
    assert_close(got, ref, "bf16", "decode MQA long")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("h_kv", [8, 2])
def test_decode_ignores_cache_rows_past_the_length(d, h_kv):
    """Cache rows at or past L_b are not part of the step (itwiki.kr "멀티 헤드 어텐션",
    section 추론 비용과 변형: the cache holds the earlier tokens); they may hold anything, here
    NaN, and the output must neither see them nor turn NaN (every case runs on the tensor-core
    decode kernel, which zeroes those V rows before the PV product and masks those keys)."""
    h, Tq = 8, 1
    B, Tmax = 3, 700
    lengths = [Tmax, 130, 513]
    Q = wl.random_tensor((B, Tq, h * d), 85, "bf16")
    Kc = wl.random_tensor((B, Tmax, h_kv * d), 86, "bf16")
    Vc = wl.random_tensor((B, Tmax, h_kv * d), 87, "bf16")
    Kn, Vn = Kc.copy(), Vc.copy()
    for b, L in enumerate(lengths):
        Kn[b, L:] = np.nan
        Vn[b, L:] = np.nan
    layer = Mha(h * d, h, d, d, dtype=torch.bfloat16, h_kv=h_kv)
    lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    O = layer.decode(to_device(Q, "bf16"), to_device(Kn, "bf16"), to_device(Vn, "bf16"), lens)
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = to_host(O)
    assert np.isfinite(got).all()
    assert_close(got, oracle.decode(Q, Kc, Vc, h, lengths, h_kv=h_kv), "bf16", "decode NaN tail")


def test_decode_split_where_early_tokens_see_no_key():
    """Several new tokens, MQA: with L = 258 the split that starts at key 256 holds no key
    visible to new tokens 0 and 1 (they see keys up to 254 and 255); their records for that
    split must carry no weight in the merge."""
    h, h_kv, d, Tq = 16, 1, 64, 4
    B, Tmax = 1, 1024
    layer, got, ref = _decode_case(88, "bf16", B, Tq, Tmax, h, h_kv, d, [258])
    assert layer.status() == 0
    assert np.isfinite(got).all()
    assert_close(got, ref, "bf16", "decode split without visible keys")
