"""Pins of the oracle's variants: residual, grouped K/V heads (MQA/GQA), the output
gate, and the KV-cache decode step (CPU only).

Each variant is tied to something other than its own formula:
  * residual (iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", sections 14
    and 16): with W^O = 0 and b^O = 0 the output is the residual exactly, and the
    residual forward minus the residual is the (already pinned) plain forward;
  * grouped heads (itwiki.kr "멀티 헤드 어텐션", 추론 비용과 변형): equal to plain MHA
    with each group's K/V projection block copied to every query head of the group,
    and to torch's scaled_dot_product_attention with enable_gqa in fp64;
  * gate (same section): a zero gate pre-activation halves every head's output, a
    saturated one leaves it unchanged, and a per-head gate equals scaling that head's
    rows of W^O;
  * decode (same section, KV cache): each new token's row equals the matching row of
    causal self-attention over the cached prefix, and torch's SDPA with a lower-right
    causal mask.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _layer(rng, B, Tq, D, h, dk, dv, h_kv=None, gated=False, Tkv=None, cross=False):
    from oracle import proj_width
    h_kv = h if h_kv is None else h_kv
    Tkv = Tq if Tkv is None else Tkv
    width = proj_width(h, dk, dv, h_kv, gated)
    Xq = rng.standard_normal((B, Tq, D))
    Xkv = rng.standard_normal((B, Tkv, D)) if cross else None
    Wqkv = rng.standard_normal((D, width)) / math.sqrt(D)
    bqkv = rng.standard_normal(width) * 0.1
    Wo = rng.standard_normal((h * dv, D)) / math.sqrt(h * dv)
    bo = rng.standard_normal(D) * 0.1
    return Xq, Xkv, Wqkv, bqkv, Wo, bo


# ---------------------------------------------------------------- residual

def test_residual_with_zero_output_projection_is_the_residual(oracle_mod):
    rng = np.random.default_rng(11)
    Xq, _, Wqkv, bqkv, Wo, bo = _layer(rng, 2, 6, 16, 4, 4, 4)
    R = rng.standard_normal(Xq.shape)
    Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, np.zeros_like(Wo), np.zeros_like(bo), 4, 4, 4,
                               causal=True, residual=R)
    np.testing.assert_array_equal(Y, R)


@pytest.mark.parametrize("causal", [False, True])
def test_residual_adds_to_the_plain_forward(oracle_mod, causal):
    rng = np.random.default_rng(12)
    Xq, _, Wqkv, bqkv, Wo, bo = _layer(rng, 2, 7, 24, 3, 8, 8)
    Y0 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, 3, 8, 8, causal=causal)
    Y1 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, 3, 8, 8, causal=causal, residual=Xq)
    np.testing.assert_allclose(Y1 - Xq, Y0, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- grouped K/V heads

def _expand_groups(Wqkv, bqkv, D, h, h_kv, dk, dv):
    """The plain-MHA weights that give every query head its group's K/V block."""
    hq, hk = h * dk, h_kv * dk
    Wq, Wk, Wv = Wqkv[:, :hq], Wqkv[:, hq:hq + hk], Wqkv[:, hq + hk:]
    bq, bk, bv = bqkv[:hq], bqkv[hq:hq + hk], bqkv[hq + hk:]
    per = h // h_kv
    Wk_e = np.concatenate([Wk[:, (i // per) * dk:(i // per + 1) * dk] for i in range(h)], axis=1)
    Wv_e = np.concatenate([Wv[:, (i // per) * dv:(i // per + 1) * dv] for i in range(h)], axis=1)
    bk_e = np.concatenate([bk[(i // per) * dk:(i // per + 1) * dk] for i in range(h)])
    bv_e = np.concatenate([bv[(i // per) * dv:(i // per + 1) * dv] for i in range(h)])
    return np.concatenate([Wq, Wk_e, Wv_e], axis=1), np.concatenate([bq, bk_e, bv_e])


@pytest.mark.parametrize("h_kv", [1, 2, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_equal_mha_with_copied_kv_blocks(oracle_mod, h_kv, causal):
    rng = np.random.default_rng(20 + h_kv)
    h, dk, dv, D = 6, 4, 4, 24
    Xq, _, Wqkv, bqkv, Wo, bo = _layer(rng, 2, 9, D, h, dk, dv, h_kv=h_kv)
    Yg = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, causal=causal, h_kv=h_kv)
    We, be = _expand_groups(Wqkv, bqkv, D, h, h_kv, dk, dv)
    Ym = oracle_mod.mha_forward(Xq, We, be, Wo, bo, h, dk, dv, causal=causal)
    np.testing.assert_allclose(Yg, Ym, rtol=0, atol=1e-13)


@pytest.mark.parametrize("h_kv", [1, 2])
def test_grouped_attention_matches_torch_sdpa_gqa_fp64(oracle_mod, h_kv):
    """torch's scaled_dot_product_attention with enable_gqa (written by others)."""
    rng = np.random.default_rng(30 + h_kv)
    B, T, h, dk = 2, 10, 4, 8
    Q = rng.standard_normal((B, T, h * dk))
    K = rng.standard_normal((B, T, h_kv * dk))
    V = rng.standard_normal((B, T, h_kv * dk))
    O = oracle_mod.attention(Q, K, V, h=h, causal=True, h_kv=h_kv)
    q = torch.from_numpy(Q).view(B, T, h, dk).transpose(1, 2)
    k = torch.from_numpy(K).view(B, T, h_kv, dk).transpose(1, 2)
    v = torch.from_numpy(V).view(B, T, h_kv, dk).transpose(1, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    ref = ref.transpose(1, 2).reshape(B, T, h * dk).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


def test_grouped_heads_reject_non_divisor(oracle_mod):
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((1, 3, 12))
    K = rng.standard_normal((1, 3, 8))
    with pytest.raises(ValueError):
        oracle_mod.attention(Q, K, K, h=3, h_kv=2)


# ---------------------------------------------------------------- gate

def _gate_layer(rng, D, h, dk, dv, gate_bias):
    """Weights with a zero gate projection and the given gate biases (per column)."""
    Xq, _, Wqkv, bqkv, Wo, bo = _layer(rng, 2, 8, D, h, dk, dv, gated=True)
    hv = h * dv
    Wqkv[:, -hv:] = 0.0
    bqkv[-hv:] = gate_bias
    return Xq, Wqkv, bqkv, Wo, bo


@pytest.mark.parametrize("causal", [False, True])
def test_zero_gate_halves_and_saturated_gate_keeps(oracle_mod, causal):
    rng = np.random.default_rng(40)
    D, h, dk, dv = 16, 2, 8, 8
    Xq, Wqkv, bqkv, Wo, bo = _gate_layer(rng, D, h, dk, dv, 0.0)
    plain_W, plain_b = Wqkv[:, :-h * dv], bqkv[:-h * dv]
    Y0 = oracle_mod.mha_forward(Xq, plain_W, plain_b, Wo, bo, h, dk, dv, causal=causal)
    Yh = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, causal=causal, gated=True)
    np.testing.assert_allclose(Yh - bo, 0.5 * (Y0 - bo), rtol=0, atol=1e-13)
    bqkv[-h * dv:] = 40.0  # sigmoid(40) = 1 - 4e-18
    Y1 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, causal=causal, gated=True)
    np.testing.assert_allclose(Y1, Y0, rtol=0, atol=1e-13)


def test_gate_is_head_specific(oracle_mod):
    """Head 0 gated at 0.5, head 1 open: equals the plain forward with head 0's rows
    of W^O halved (so the gate multiplies head 0's output columns, not head 1's)."""
    rng = np.random.default_rng(41)
    D, h, dk, dv = 16, 2, 8, 8
    gb = np.concatenate([np.zeros(dv), np.full(dv, 40.0)])
    Xq, Wqkv, bqkv, Wo, bo = _gate_layer(rng, D, h, dk, dv, gb)
    Yg = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, causal=True, gated=True)
    Wo2 = Wo.copy()
    Wo2[:dv] *= 0.5
    Y2 = oracle_mod.mha_forward(Xq, Wqkv[:, :-h * dv], bqkv[:-h * dv], Wo2, bo, h, dk, dv, causal=True)
    np.testing.assert_allclose(Yg, Y2, rtol=0, atol=1e-13)


def test_gate_uses_the_logistic_function(oracle_mod):
    """A gate pre-activation of log(3) gives 3/4: 1/(1+e^-x), not e.g. tanh or a
    sign slip (1/(1+e^x) would give 1/4)."""
    rng = np.random.default_rng(42)
    D, h, dk, dv = 8, 1, 8, 8
    Xq, Wqkv, bqkv, Wo, bo = _gate_layer(rng, D, h, dk, dv, math.log(3.0))
    Y0 = oracle_mod.mha_forward(Xq, Wqkv[:, :-dv], bqkv[:-dv], Wo, bo, h, dk, dv)
    Yg = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, gated=True)
    np.testing.assert_allclose(Yg - bo, 0.75 * (Y0 - bo), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("Tq", [1, 3])
@pytest.mark.parametrize("h_kv", [4, 2, 1])
def test_decode_rows_equal_causal_self_attention_rows(oracle_mod, Tq, h_kv):
    rng = np.random.default_rng(50 + Tq + h_kv)
    B, Tmax, h, dk = 3, 12, 4, 8
    lens = np.array([12, 5, 3], dtype=np.int32)
    Kc = rng.standard_normal((B, Tmax, h_kv * dk))
    Vc = rng.standard_normal((B, Tmax, h_kv * dk))
    Q = rng.standard_normal((B, Tq, h * dk))
    O = oracle_mod.decode(Q, Kc, Vc, h, lens, h_kv=h_kv)
    for b in range(B):
        L = int(lens[b])
        Qfull = np.zeros((1, L, h * dk))
        Qfull[0, L - Tq:] = Q[b]
        ref = oracle_mod.attention(Qfull, Kc[b:b + 1, :L], Vc[b:b + 1, :L], h=h, causal=True, h_kv=h_kv)
        np.testing.assert_allclose(O[b], ref[0, L - Tq:], rtol=0, atol=1e-13)


def test_decode_matches_torch_sdpa_lower_right_mask(oracle_mod):
    rng = np.random.default_rng(60)
    B, Tq, Tmax, h, dk = 1, 4, 9, 2, 8
    Kc = rng.standard_normal((B, Tmax, h * dk))
    Vc = rng.standard_normal((B, Tmax, h * dk))
    Q = rng.standard_normal((B, Tq, h * dk))
    O = oracle_mod.decode(Q, Kc, Vc, h, [Tmax])
    q = torch.from_numpy(Q).view(B, Tq, h, dk).transpose(1, 2)
    k = torch.from_numpy(Kc).view(B, Tmax, h, dk).transpose(1, 2)
    v = torch.from_numpy(Vc).view(B, Tmax, h, dk).transpose(1, 2)
    # new token t sits at position Tmax - Tq + t: keys after it are hidden
    allowed = torch.ones(Tq, Tmax, dtype=torch.bool).tril(diagonal=Tmax - Tq)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed)
    ref = ref.transpose(1, 2).reshape(B, Tq, h * dk).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


def test_decode_invalid_lengths_give_nan_rows(oracle_mod):
    rng = np.random.default_rng(61)
    B, Tq, Tmax, h, dk = 3, 2, 6, 2, 4
    Kc = rng.standard_normal((B, Tmax, h * dk))
    Q = rng.standard_normal((B, Tq, h * dk))
    O = oracle_mod.decode(Q, Kc, Kc, h, [1, 7, 6])  # L < Tq, L > Tmax, valid
    assert np.isnan(O[0]).all() and np.isnan(O[1]).all()
    assert np.isfinite(O[2]).all()
