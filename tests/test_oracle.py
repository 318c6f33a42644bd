"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Every test here runs on the CPU (no ``gpu`` mark).  Each pin is chosen so that
a plausible slip in the oracle -- a wrong scale, a dropped bias, a transposed
weight, a wrong head slice or concat index, a mask off by one, a softmax over
the wrong axis -- fails at least one of them:

  * closed forms (two keys; zero queries give the uniform mean of the values);
  * invariants the pages state (rows of the weights sum to 1 and are >= 0;
    masked weights are exactly 0; parameters 4E^2 + 4E whatever the head
    count; h heads of width d_v concatenate to h*d_v);
  * reductions to library routines written by others (torch's
    scaled_dot_product_attention and nn.MultiheadAttention, in fp64 on CPU;
    scipy's softmax for the single-head case);
  * brute force on tiny inputs, and symmetries (head and sequence
    permutations).
"""
import json
import math
import os

import numpy as np
import pytest

from transformer_head_scaled_02_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_layer(rng, B, Tq, D, h, dk, dv, Tkv=None, bias=True, cross=False):
    Tkv = Tq if Tkv is None else Tkv
    Xq = rng.standard_normal((B, Tq, D))
    Xkv = rng.standard_normal((B, Tkv, D)) if cross else None
    Wqkv = rng.standard_normal((D, 2 * h * dk + h * dv)) / math.sqrt(D)
    Wo = rng.standard_normal((h * dv, D)) / math.sqrt(h * dv)
    bqkv = rng.standard_normal(2 * h * dk + h * dv) * 0.1 if bias else None
    bo = rng.standard_normal(D) * 0.1 if bias else None
    return Xq, Xkv, Wqkv, bqkv, Wo, bo


# ---------------------------------------------------------------- closed forms

def test_two_key_closed_form_fixes_scale(oracle_mod):
    """q=(2,0,0,0), k0=(1,0,0,0), k1=0, d_k=4: the scores are 2/sqrt(4)=1 and 0,
    so the weights are e/(e+1) and 1/(e+1).  A scale of 1/d_k (the garbled
    formula on wiki.railscraft.dev) would give e^0.5/(e^0.5+1) instead; the
    scale 1/sqrt(d_k) is the one of itwiki.kr "멀티 헤드 어텐션", 수식."""
    Q = np.array([[[2.0, 0, 0, 0]]])
    K = np.array([[[1.0, 0, 0, 0], [0.0, 0, 0, 0]]])
    V = np.array([[[1.0, 0, 0, 0], [0.0, 1, 0, 0]]])
    O, P = oracle_mod.attention(Q, K, V, h=1, return_weights=True)
    e = math.e
    assert P[0, 0, 0, 0] == pytest.approx(e / (e + 1), rel=1e-15, abs=0)
    assert P[0, 0, 0, 1] == pytest.approx(1 / (e + 1), rel=1e-15, abs=0)
    np.testing.assert_allclose(O[0, 0], [e / (e + 1), 1 / (e + 1), 0, 0], rtol=1e-15, atol=0)


def test_zero_queries_give_uniform_mean_of_values(oracle_mod):
    """With W_Q = 0 and b_Q = 0 every score is 0, so each head averages the
    value rows it may see: all of them, the first t+1 under the causal mask,
    the first L_b under key padding.  Closed form, computed with numpy."""
    rng = np.random.default_rng(1)
    B, T, D, h, dk = 2, 7, 12, 3, 4
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dk)
    Wqkv[:, : h * dk] = 0.0
    bqkv[: h * dk] = 0.0
    Vf = Xq @ Wqkv[:, 2 * h * dk:] + bqkv[2 * h * dk:]
    for causal, kvl in ((False, None), (True, None), (False, np.array([3, 7]))):
        Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, causal=causal,
                                   kv_lengths=kvl)
        O = np.empty((B, T, h * dk))
        for b in range(B):
            for t in range(T):
                n = t + 1 if causal else (kvl[b] if kvl is not None else T)
                O[b, t] = Vf[b, :n].mean(axis=0)
        np.testing.assert_allclose(Y, O @ Wo + bo, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_weight_rows_sum_to_one_and_are_nonnegative(oracle_mod, causal):
    """iamjaehka13.blog, section 10: A_ij >= 0 and sum_j A_ij = 1."""
    rng = np.random.default_rng(2)
    B, T, h, dk = 2, 9, 3, 5
    Q = rng.standard_normal((B, T, h * dk)) * 3
    K = rng.standard_normal((B, T, h * dk)) * 3
    V = rng.standard_normal((B, T, h * dk))
    _, P = oracle_mod.attention(Q, K, V, h=h, causal=causal, return_weights=True)
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, rtol=0, atol=1e-14)


def test_causal_weights_are_exactly_zero_above_diagonal(oracle_mod):
    """iamjaehka13.blog, section 9: masked scores are -inf, so their weights
    are exactly exp(-inf) = 0, not merely small; j <= i stays positive."""
    rng = np.random.default_rng(3)
    B, T, h, dk = 2, 11, 2, 4
    Q, K, V = (rng.standard_normal((B, T, h * dk)) for _ in range(3))
    _, P = oracle_mod.attention(Q, K, V, h=h, causal=True, return_weights=True)
    iu = np.triu_indices(T, 1)
    assert (P[..., iu[0], iu[1]] == 0.0).all()
    il = np.tril_indices(T)
    assert (P[..., il[0], il[1]] > 0.0).all()


def test_padding_weights_zero_and_padded_rows_do_not_matter(oracle_mod):
    """molayo1419.me, pitfall 2: keys marked as padding are not read.  Their
    weights are exactly 0 and the output does not change, bit for bit, when
    the padded rows of the key/value states are replaced by anything finite."""
    rng = np.random.default_rng(4)
    B, Tq, Tkv, D, h, dk = 3, 5, 9, 8, 2, 4
    Xq, Xkv, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, Tq, D, h, dk, dk, Tkv=Tkv, cross=True)
    kvl = np.array([1, 4, 9], dtype=np.int32)
    Y1 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, Xkv=Xkv, kv_lengths=kvl)
    Xkv2 = Xkv.copy()
    for b in range(B):
        Xkv2[b, kvl[b]:] = rng.standard_normal((Tkv - kvl[b], D)) * 1e3
    Y2 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, Xkv=Xkv2, kv_lengths=kvl)
    assert np.array_equal(Y1, Y2)
    Q = Xq @ Wqkv[:, : h * dk]
    K = Xkv @ Wqkv[:, h * dk: 2 * h * dk]
    V = Xkv @ Wqkv[:, 2 * h * dk:]
    _, P = oracle_mod.attention(Q, K, V, h=h, kv_lengths=kvl, return_weights=True)
    for b in range(B):
        assert (P[b, ..., kvl[b]:] == 0.0).all()
        assert (P[b, ..., : kvl[b]] > 0.0).all()


def test_all_keys_masked_gives_nan(oracle_mod):
    """molayo1419.me, pitfall 3: when every key of a sample is ignored the
    softmax is 0/0 and the output is NaN (in training and eval mode alike).
    The other samples are unaffected."""
    rng = np.random.default_rng(5)
    B, T, D, h, dk = 2, 4, 8, 2, 4
    Xq, Xkv, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dk, cross=True)
    Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, Xkv=Xkv,
                               kv_lengths=np.array([0, 3]))
    assert np.isnan(Y[0]).all()
    assert np.isfinite(Y[1]).all()


def test_parameter_count_independent_of_heads(oracle_mod):
    """Golden: molayo1419.me parameter table -- E = 512 gives 1,050,624
    parameters for any head count.  The count is taken from the shapes the
    oracle accepts (it rejects any other), with d_k = d_v = E/h as on the
    page; the oracle runs once per head count so the shapes are live."""
    with open(os.path.join(GOLDEN, "param_count_e512.json")) as f:
        g = json.load(f)
    E = g["E"]
    rng = np.random.default_rng(6)
    X = rng.standard_normal((1, 2, E))
    for h in g["num_heads"]:
        d = E // h
        Wqkv = np.zeros((E, 3 * E))
        bqkv = np.zeros(3 * E)
        Wo = np.zeros((E, E))
        bo = np.zeros(E)
        Y = oracle_mod.mha_forward(X, Wqkv, bqkv, Wo, bo, h, d, d)
        assert Y.shape == (1, 2, E)
        assert Wqkv.size + bqkv.size + Wo.size + bo.size == g["parameter_count"]
        with pytest.raises(ValueError):
            oracle_mod.mha_forward(X, np.zeros((E, 3 * E + 1)), None, Wo, None, h, d, d)


def test_concat_width_worked_example(oracle_mod):
    """Golden: wiki.railscraft.dev worked example, 8 heads of d_v = 4 give a
    32-wide concatenation; each head's output lands in its own 4 columns."""
    with open(os.path.join(GOLDEN, "concat_width_h8_dv4.json")) as f:
        g = json.load(f)
    h, dv = g["h"], g["d_v"]
    rng = np.random.default_rng(7)
    B, T, dk = 1, 16, 4
    Q = rng.standard_normal((B, T, h * dk))
    K = rng.standard_normal((B, T, h * dk))
    V = np.zeros((B, T, h * dv))
    head = 5
    V[..., head * dv:(head + 1) * dv] = 1.0       # only head 5 has nonzero values
    O = oracle_mod.attention(Q, K, V, h=h)
    assert O.shape[-1] == g["concat_width"]
    np.testing.assert_allclose(O[..., head * dv:(head + 1) * dv], 1.0, rtol=1e-14)
    mask = np.ones(h * dv, bool)
    mask[head * dv:(head + 1) * dv] = False
    assert (O[..., mask] == 0.0).all()


# ---------------------------------------------------------------- library reductions

def _torch():
    return pytest.importorskip("torch")


@pytest.mark.parametrize("causal,padded", [(False, False), (True, False), (False, True)])
def test_matches_torch_sdpa_fp64(oracle_mod, causal, padded):
    """Per-head attention equals torch.nn.functional.scaled_dot_product_attention
    (itwiki.kr "멀티 헤드 어텐션", 구현: the library routine for the same
    softmax(QK^T/sqrt(d_k))V), run in fp64 on CPU on the same projected
    inputs.  The projections themselves are checked with numpy matmul."""
    torch = _torch()
    rng = np.random.default_rng(8)
    B, Tq, D, h, dk = 2, 13, 24, 3, 8
    Tkv = Tq if not padded else 17
    cross = padded
    Xq, Xkv, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, Tq, D, h, dk, dk, Tkv=Tkv, cross=cross)
    kvl = np.array([5, 17], dtype=np.int32) if padded else None
    Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, Xkv=Xkv, causal=causal,
                               kv_lengths=kvl)
    src = Xq if Xkv is None else Xkv
    q = torch.from_numpy(Xq @ Wqkv[:, :h * dk] + bqkv[:h * dk])
    k = torch.from_numpy(src @ Wqkv[:, h * dk:2 * h * dk] + bqkv[h * dk:2 * h * dk])
    v = torch.from_numpy(src @ Wqkv[:, 2 * h * dk:] + bqkv[2 * h * dk:])
    q, k, v = (t.view(B, t.shape[1], h, dk).transpose(1, 2) for t in (q, k, v))
    mask = None
    if causal:
        mask = torch.ones(Tq, Tkv, dtype=torch.bool).tril()
    if padded:
        keep = torch.arange(Tkv)[None, :] < torch.from_numpy(kvl)[:, None].long()
        mask = keep[:, None, None, :].expand(B, 1, Tq, Tkv)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    o = o.transpose(1, 2).reshape(B, Tq, h * dk).numpy()
    np.testing.assert_allclose(Y, o @ Wo + bo, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_multihead_attention_fp64(oracle_mod, causal):
    """The whole layer equals torch.nn.MultiheadAttention in fp64 with
    batch_first=True (molayo1419.me shows that module is the formula itself).
    nn.Linear keeps weights as (out, in), so ours go in transposed; its
    key_padding_mask marks ignored keys with True."""
    torch = _torch()
    rng = np.random.default_rng(9)
    B, T, D, h = 3, 10, 32, 4
    dk = D // h
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dk)
    kvl = np.array([10, 6, 1], dtype=np.int32)
    Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, causal=causal,
                               kv_lengths=kvl)
    m = torch.nn.MultiheadAttention(D, h, batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        m.in_proj_weight.copy_(torch.from_numpy(Wqkv.T))
        m.in_proj_bias.copy_(torch.from_numpy(bqkv))
        m.out_proj.weight.copy_(torch.from_numpy(Wo.T))
        m.out_proj.bias.copy_(torch.from_numpy(bo))
    m.eval()
    x = torch.from_numpy(Xq)
    kpm = torch.arange(T)[None, :] >= torch.from_numpy(kvl)[:, None].long()
    am = torch.ones(T, T, dtype=torch.bool).triu(1) if causal else None
    with torch.no_grad():
        ref, _ = m(x, x, x, key_padding_mask=kpm, attn_mask=am, need_weights=False)
    np.testing.assert_allclose(Y, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_single_head_reduces_to_one_attention(oracle_mod):
    """h = 1 is the single-head layer of iamjaehka13.blog, section 16:
    softmax((X W_Q)(X W_K)^T / sqrt(d_k) + M) (X W_V) W_O, here written with
    numpy matmuls and scipy's softmax."""
    from scipy.special import softmax
    rng = np.random.default_rng(10)
    B, T, D = 2, 8, 6
    dk = 5
    Xq, _, Wqkv, _, Wo, _ = _rand_layer(rng, B, T, D, 1, dk, dk, bias=False)
    for causal in (False, True):
        Y = oracle_mod.mha_forward(Xq, Wqkv, None, Wo, None, 1, dk, dk, causal=causal)
        M = np.where(np.triu(np.ones((T, T)), 1) > 0, -np.inf, 0.0) if causal else 0.0
        for b in range(B):
            X = Xq[b]
            S = (X @ Wqkv[:, :dk]) @ (X @ Wqkv[:, dk:2 * dk]).T / math.sqrt(dk) + M
            ref = softmax(S, axis=-1) @ (X @ Wqkv[:, 2 * dk:]) @ Wo
            np.testing.assert_allclose(Y[b], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- brute force

def test_brute_force_tiny(oracle_mod):
    """T <= 4: every output element enumerated with scalar Python arithmetic,
    head by head, straight from the composition MultiHead = Concat(head_i) W^O,
    head_i = softmax(Q_i K_i^T / sqrt(d_k) + M) V_i, Q_i = X W_i^Q + b."""
    rng = np.random.default_rng(11)
    B, T, D, h, dk, dv = 2, 4, 5, 2, 3, 2
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dv)
    for causal in (False, True):
        Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, causal=causal)
        for b in range(B):
            cat = [[0.0] * (h * dv) for _ in range(T)]
            for i in range(h):
                def proj(t, col0, width):
                    return [math.fsum(Xq[b, t, c] * Wqkv[c, col0 + e] for c in range(D))
                            + bqkv[col0 + e] for e in range(width)]
                q = [proj(t, i * dk, dk) for t in range(T)]
                k = [proj(t, h * dk + i * dk, dk) for t in range(T)]
                v = [proj(t, 2 * h * dk + i * dv, dv) for t in range(T)]
                for t in range(T):
                    keys = range(t + 1) if causal else range(T)
                    s = {j: math.fsum(q[t][e] * k[j][e] for e in range(dk)) / math.sqrt(dk)
                         for j in keys}
                    z = math.fsum(math.exp(x) for x in s.values())
                    for e in range(dv):
                        cat[t][i * dv + e] = math.fsum(math.exp(s[j]) / z * v[j][e] for j in keys)
            for t in range(T):
                for n in range(D):
                    ref = math.fsum(cat[t][c] * Wo[c, n] for c in range(h * dv)) + bo[n]
                    assert Y[b, t, n] == pytest.approx(ref, rel=1e-12, abs=1e-13)


# ---------------------------------------------------------------- symmetries

def test_head_permutation_leaves_output_unchanged(oracle_mod):
    """Heads are independent (wiki.railscraft.dev: each head is its own matrix
    computation); permuting them together with their W^Q, W^K, W^V column
    slices and their W^O row slices must not change the output."""
    rng = np.random.default_rng(12)
    B, T, D, h, dk, dv = 2, 6, 10, 4, 3, 5
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dv)
    perm = np.array([2, 0, 3, 1])

    def cols(base, width):
        return np.concatenate([np.arange(base + p * width, base + (p + 1) * width) for p in perm])

    c = np.concatenate([cols(0, dk), cols(h * dk, dk), cols(2 * h * dk, dv)])
    Y1 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dv, causal=True)
    Y2 = oracle_mod.mha_forward(Xq, Wqkv[:, c], bqkv[c], Wo[cols(0, dv)], bo, h, dk, dv,
                                causal=True)
    np.testing.assert_allclose(Y1, Y2, rtol=1e-12, atol=1e-13)


def test_sequence_permutation_equivariance(oracle_mod):
    """Without a causal mask self-attention has no notion of position:
    permuting the tokens permutes the output rows the same way."""
    rng = np.random.default_rng(13)
    B, T, D, h, dk = 2, 9, 8, 2, 4
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dk)
    perm = rng.permutation(T)
    Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk)
    Yp = oracle_mod.mha_forward(Xq[:, perm], Wqkv, bqkv, Wo, bo, h, dk, dk)
    np.testing.assert_allclose(Yp, Y[:, perm], rtol=1e-12, atol=1e-13)


def test_sampled_rows_equal_full_rows(oracle_mod):
    """Computing only some query rows gives bit-identical rows to the full run
    (the sampled mode is what full-size parity checks use)."""
    rng = np.random.default_rng(14)
    B, T, D, h, dk = 2, 20, 16, 4, 4
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, B, T, D, h, dk, dk)
    rows = np.array([0, 1, 7, 19])
    kvl = np.array([20, 9])
    for causal in (False, True):
        Y = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, causal=causal, kv_lengths=kvl)
        Ys = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, h, dk, dk, causal=causal,
                                    kv_lengths=kvl, rows=rows)
        assert np.array_equal(Ys, Y[:, rows])


def test_thread_count_does_not_change_results(oracle_mod):
    rng = np.random.default_rng(15)
    Xq, _, Wqkv, bqkv, Wo, bo = _rand_layer(rng, 2, 33, 16, 4, 4, 4)
    Y1 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, 4, 4, 4, causal=True, nthreads=1)
    Y4 = oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, 4, 4, 4, causal=True, nthreads=4)
    assert np.array_equal(Y1, Y4)


def test_rejects_causal_cross_and_bad_rows(oracle_mod):
    rng = np.random.default_rng(16)
    Xq, Xkv, Wqkv, bqkv, Wo, bo = _rand_layer(rng, 1, 3, 4, 1, 4, 4, Tkv=5, cross=True)
    with pytest.raises(ValueError):
        oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, 1, 4, 4, Xkv=Xkv, causal=True)
    with pytest.raises(ValueError):
        oracle_mod.mha_forward(Xq, Wqkv, bqkv, Wo, bo, 1, 4, 4, rows=[3])


# ---------------------------------------------------------------- input generator

def test_bf16_rounding_matches_torch():
    """The shared input generator's bf16 rounding is round-to-nearest-even,
    the same as torch's float32 -> bfloat16 conversion."""
    torch = _torch()
    rng = np.random.default_rng(17)
    a = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 3.3895e38,
                                  np.inf, -np.inf], dtype=np.float32)])
    ours = wl.bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- rounded diagnostic mode

def test_oracle_bf16_rounding_ties_to_even_and_matches_torch(oracle_mod):
    """The rounded mode's own bf16 rounding: ties go to the even neighbour, and on float32
    inputs it agrees with torch's float32 -> bfloat16 conversion bit for bit."""
    r = oracle_mod.round_bf16
    assert r(1.0 + 2.0 ** -8) == 1.0                      # tie, 1.0 is even
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6      # tie, 1 + 2^-6 is even
    assert r(-(1.0 + 2.0 ** -8 + 2.0 ** -20)) == -(1.0 + 2.0 ** -7)  # just above a tie
    assert r(0.0) == 0.0 and r(2.0 ** -100) == 2.0 ** -100
    torch = _torch()
    rng = np.random.default_rng(23)
    a = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([r(float(v)) for v in a])
    assert np.array_equal(got, ref)


def test_rounded_mode_rounds_the_weights_but_not_their_sum(oracle_mod):
    """One query, two keys, d = 1, every projection exact: scores 1 and 1.5, so the
    unnormalised weights are e^-0.5 and 1.  The rounded mode divides bf16(e^-0.5) * v_0 +
    1 * v_1 by the unrounded sum e^-0.5 + 1 and rounds the result; the plain mode is the
    textbook value."""
    Xq = np.array([[[1.0]]])
    Xkv = np.array([[[1.0], [1.5]]])
    Wqkv = np.array([[1.0, 1.0, 1.0]])  # Q = x, K = x, V = x
    Wo = np.array([[1.0]])
    kw = dict(h=1, d_k=1, d_v=1, Xkv=Xkv)
    p0 = math.exp(-0.5)
    plain = oracle_mod.mha_forward(Xq, Wqkv, None, Wo, None, **kw)
    rounded = oracle_mod.mha_forward(Xq, Wqkv, None, Wo, None, round_bf16=True, **kw)
    assert plain[0, 0, 0] == pytest.approx((p0 * 1.0 + 1.5) / (p0 + 1.0), rel=1e-15)
    p0_bf16 = float(wl.round_to_bf16(np.array([p0], dtype=np.float32))[0])
    assert p0_bf16 != p0
    o = (p0_bf16 * 1.0 + 1.5) / (p0 + 1.0)
    o_bf16 = float(wl.round_to_bf16(np.array([o], dtype=np.float32))[0])
    assert rounded[0, 0, 0] == o_bf16


def test_rounded_mode_is_exact_when_nothing_needs_rounding(oracle_mod):
    """Small integers everywhere and one key per query: every stored value is a bf16 number,
    so the rounded mode equals the plain forward exactly."""
    rng = np.random.default_rng(29)
    Xq = rng.integers(-3, 4, (2, 1, 8)).astype(np.float64)
    Wqkv = rng.integers(-1, 2, (8, 24)).astype(np.float64)
    Wo = rng.integers(-1, 2, (8, 8)).astype(np.float64)
    bq = rng.integers(-2, 3, 24).astype(np.float64)
    plain = oracle_mod.mha_forward(Xq, Wqkv, bq, Wo, None, h=2, d_k=4, d_v=4)
    rounded = oracle_mod.mha_forward(Xq, Wqkv, bq, Wo, None, h=2, d_k=4, d_v=4, round_bf16=True)
    assert np.array_equal(plain, rounded)


def test_rounded_mode_stays_within_the_bf16_budget(oracle_mod):
    """On bf16 inputs the rounded forward differs from the plain one by about the bf16
    storage error: more than nothing, well under the parity bound."""
    w = wl.custom("rounded", B=2, T_q=70, D=128, h=2, d_k=64, causal=True)
    x = wl.make_inputs(w, seed=4)
    args = (x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h, w.d_k, w.d_v)
    plain = oracle_mod.mha_forward(*args, causal=True)
    rounded = oracle_mod.mha_forward(*args, causal=True, round_bf16=True)
    rel = np.linalg.norm(rounded - plain) / np.linalg.norm(plain)
    assert 5e-4 < rel < 5e-3
    # Y itself is bf16: every rounded output is a bf16 number
    assert np.array_equal(rounded.astype(np.float32), wl.round_to_bf16(rounded.astype(np.float32)))


def test_named_workloads_are_seeded_and_shaped():
    for name, w in wl.WORKLOADS.items():
        if w.B * w.T_q * w.D > 2_000_000:
            continue
        a = wl.make_inputs(w)
        b = wl.make_inputs(w)
        assert a["X_q"].shape == (w.B, w.T_q, w.D)
        assert a["W_qkv"].shape == (w.D, 2 * w.h * w.d_k + w.h * w.d_v)
        assert a["W_o"].shape == (w.h * w.d_v, w.D)
        for k in a:
            if a[k] is None:
                assert b[k] is None
            else:
                assert np.array_equal(a[k], b[k])
    f = wl.flops(wl.WORKLOADS["c3_bf16_causal"])
    assert f["total"] == pytest.approx(103.08e9, rel=1e-3)
