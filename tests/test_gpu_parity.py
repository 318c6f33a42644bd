"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs.

  * single steps: the projection GEMM (mha_linear) and the fused attention
    (mha_attention) against the oracle's linear / attention steps, element by
    element, over shapes that span several tiles and a ragged tail;
  * the whole forward (mha_forward) on small shapes, element by element,
    including cross-attention with key padding, d = 64 and 128, fp32 and bf16;
  * the five named workloads at full size, every output element;
  * edge cases: empty batch, one query row, one valid key, invalid lengths
    (NaN rows and a device status), guard bands around the output, padding
    invariance, determinism.
Tolerances are those of tests/gpu_util.py.
"""
import numpy as np
import pytest

from gpu_util import assert_close, errors, to_device, to_host, torch_dtype

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


def _layer(w):
    return Mha(w.D, w.h, w.d_k, w.d_v, dtype=torch_dtype(w.dtype))


def _run_forward(w, x, layer=None):
    layer = layer or _layer(w)
    d = {k: to_device(v, w.dtype) for k, v in x.items() if k != "kv_lengths"}
    kvl = None if x["kv_lengths"] is None else torch.from_numpy(x["kv_lengths"]).cuda()
    y = layer.forward(d["X_q"], d["W_qkv"], d["b_qkv"], d["W_o"], d["b_o"], X_kv=d["X_kv"],
                      causal=w.causal, kv_lengths=kvl)
    torch.cuda.synchronize()
    return layer, y


def _oracle_forward(w, x, rows=None):
    return oracle.mha_forward(x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h, w.d_k,
                              w.d_v, Xkv=x["X_kv"], causal=w.causal, kv_lengths=x["kv_lengths"],
                              rows=rows)


# ------------------------------------------------------------------ step: projection GEMM

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M,K,N,bias", [
    (1, 64, 64, True),          # one row
    (300, 1024, 3072, True),    # ragged M, several N tiles
    (257, 72, 200, False),      # K tail inside a 64-wide block, N tail inside a 256-wide tile
    (300, 64, 256, True),       # one 64-wide K half: the second half of the stage is skipped
    (260, 192, 520, False),     # K = 1.5 stages of 128
    (1024, 512, 1536, True),
])
def test_linear_step(dtype, M, K, N, bias):
    A = wl.random_tensor((M, K), seed=1, dtype=dtype)
    W = wl.random_tensor((K, N), seed=2, dtype=dtype, scale=0.05)
    b = wl.random_tensor((N,), seed=3, dtype=dtype, scale=0.1) if bias else None
    layer = Mha(64, 1, 64, dtype=torch_dtype(dtype))
    C = layer.linear(to_device(A, dtype), to_device(W, dtype), to_device(b, dtype))
    torch.cuda.synchronize()
    assert_close(to_host(C), oracle.linear(A, W, b), dtype, f"linear {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N,residual", [
    (32, 1024, 3072, False),    # a decode step's QKV projection: 24 tiles, clusters of 4
    (100, 1032, 520, True),     # K tail inside a 64-wide block, N tail; 6 ranks of 3 K blocks
    (128, 4096, 1024, True),    # 8 tiles, 8 ranks of 8 K blocks
    (1, 2048, 12288, False),    # one row; 96 tiles of 128 columns: 48 of 256 in clusters of 2
    (7, 136, 264, False),       # three K blocks over three ranks; N tail
    (64, 512, 16384, True),     # 64 tiles of 256 columns in clusters of 2
    (16, 512, 33024, False),    # 129 tiles of 256 columns: one CTA per tile
])
def test_linear_step_bf16_few_rows(M, K, N, residual):
    """bf16 projections of at most 128 rows, where clusters of CTAs split K and add their
    partial tiles through distributed shared memory: C = A W + bias (+ R) equals the oracle's
    (the residual form adds R in the same epilogue), and a second call gives the same bits (the
    partials are added in rank order)."""
    A = wl.random_tensor((M, K), seed=41, dtype="bf16")
    W = wl.random_tensor((K, N), seed=42, dtype="bf16", scale=0.5 / np.sqrt(K))
    b = wl.random_tensor((N,), seed=43, dtype="bf16", scale=0.1)
    R = wl.random_tensor((M, N), seed=44, dtype="bf16") if residual else None
    layer = Mha(64, 1, 64, dtype=torch.bfloat16)
    layer.ensure_workspace(1, 1, 1)
    Ad, Wd, bd, Rd = (to_device(t, "bf16") for t in (A, W, b, R))
    C1 = layer.linear(Ad, Wd, bd, residual=Rd)
    C2 = layer.linear(Ad, Wd, bd, residual=Rd)
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = oracle.linear(A, W, b)
    if residual:
        ref = ref + R.astype(np.float64)  # already bf16 values
    assert_close(to_host(C1), ref, "bf16", f"few-row linear {M}x{K}x{N}")
    assert torch.equal(C1, C2), "a second call gave a different result"


@pytest.mark.parametrize("M,K,N,residual", [
    (128, 1024, 1024, False),   # 32 tiles: K over clusters of 8
    (1024, 512, 512, True),     # 128 tiles: clusters of 4 (the fp32 causal output projection)
    (100, 296, 200, True),      # ragged K over 4 ranks (10 slices of 32: 3 + 3 + 3 + 1)
    (70, 517, 45, False),       # unaligned rows; 17 slices over 8 ranks, the last two empty
])
def test_linear_step_f32_split(M, K, N, residual):
    """fp32 projections with no more 64 x 64 tiles than SMs split K over clusters whose fp32
    partial tiles are added in rank order through distributed shared memory: C = A W + bias
    (+ R) equals the oracle's, the same bits on a second call."""
    A = wl.random_tensor((M, K), seed=51, dtype="f32")
    W = wl.random_tensor((K, N), seed=52, dtype="f32", scale=0.05)
    b = wl.random_tensor((N,), seed=53, dtype="f32", scale=0.1)
    R = wl.random_tensor((M, N), seed=54, dtype="f32") if residual else None
    layer = Mha(64, 1, 64, dtype=torch.float32)
    layer.ensure_workspace(1, 1, 1)
    Ad, Wd, bd, Rd = (to_device(t, "f32") for t in (A, W, b, R))
    C1 = layer.linear(Ad, Wd, bd, residual=Rd)
    C2 = layer.linear(Ad, Wd, bd, residual=Rd)
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = oracle.linear(A, W, b)
    if residual:
        ref = ref + R.astype(np.float64)
    assert_close(to_host(C1), ref, "f32", f"f32 split linear {M}x{K}x{N}")
    assert torch.equal(C1, C2), "a second call gave a different result"


@pytest.mark.parametrize("M,K,N", [(70, 37, 45), (129, 130, 67), (64, 33, 64)])
def test_linear_step_f32_unaligned(M, K, N):
    """fp32 projections whose row strides are not a multiple of four floats take the scalar
    global loads of the fp32 GEMM (no 16-byte loads); the sums are the same."""
    A = wl.random_tensor((M, K), seed=4, dtype="f32")
    W = wl.random_tensor((K, N), seed=5, dtype="f32", scale=0.05)
    b = wl.random_tensor((N,), seed=6, dtype="f32", scale=0.1)
    layer = Mha(64, 1, 64, dtype=torch.float32)
    C = layer.linear(to_device(A, "f32"), to_device(W, "f32"), to_device(b, "f32"))
    torch.cuda.synchronize()
    assert_close(to_host(C), oracle.linear(A, W, b), "f32", f"f32 linear {M}x{K}x{N}")


@pytest.mark.parametrize("dtype,M,M2,N,N2,K,lens", [
    ("bf16", 4 * 700, 300, 384, 200, 192, [1, 300, 700, 129]),   # one launch, segments, ragged
    ("bf16", 1000, 8192, 1536, 768, 256, None),                  # one launch, second one larger
    ("bf16", 600, 100, 256, 512, 128, None),                     # M2 <= 128: two launches
    ("f32", 4 * 700, 300, 72, 40, 48, [1, 300, 700, 129]),       # fp32: two launches
])
def test_linear_pair(dtype, M, M2, N, N2, K, lens):
    """mha_linear_pair: both outputs equal the oracle's projections (with segment lengths, the
    rows the attention step reads), whether the two run in one launch or one after the other."""
    A = wl.random_tensor((M, K), seed=31, dtype=dtype)
    W = wl.random_tensor((K, N), seed=32, dtype=dtype, scale=0.05)
    b = wl.random_tensor((N,), seed=33, dtype=dtype, scale=0.1)
    A2 = wl.random_tensor((M2, K), seed=34, dtype=dtype)
    W2 = wl.random_tensor((K, N2), seed=35, dtype=dtype, scale=0.05)
    b2 = wl.random_tensor((N2,), seed=36, dtype=dtype, scale=0.1)
    layer = Mha(64, 1, 64, dtype=torch_dtype(dtype))
    seg = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch_dtype(dtype), device="cuda")
    out2 = torch.full((M2, N2), float("nan"), dtype=torch_dtype(dtype), device="cuda")
    layer.linear_pair(to_device(A, dtype), to_device(W, dtype), to_device(b, dtype),
                      to_device(A2, dtype), to_device(W2, dtype), to_device(b2, dtype),
                      seg_len=seg, seg_rows=0 if lens is None else 700, out=out, out2=out2)
    torch.cuda.synchronize()
    assert_close(to_host(out2), oracle.linear(A2, W2, b2), dtype, "second projection")
    ref, got = oracle.linear(A, W, b), to_host(out)
    if lens is None:
        assert_close(got, ref, dtype, "first projection")
    else:
        for i, L in enumerate(lens):
            need = min((int(L) + 127) // 128 * 128, 700)
            rows = slice(i * 700, i * 700 + need)
            assert_close(got[rows], ref[rows], dtype, f"first projection, segment {i} (length {L})")


def test_linear_segments_writes_every_needed_row():
    """mha_linear_segments: the rows of each segment below its length rounded up to 128 equal
    the oracle's projection (the rest may be skipped).  Segments of 700 rows straddle the
    GEMM's 256-row blocks."""
    lens = np.array([1, 300, 700, 129], dtype=np.int32)
    seg, K, N = 700, 192, 384
    A = wl.random_tensor((len(lens) * seg, K), seed=21)
    W = wl.random_tensor((K, N), seed=22, scale=0.05)
    b = wl.random_tensor((N,), seed=23, scale=0.1)
    layer = Mha(64, 1, 64, dtype=torch.bfloat16)
    C = torch.full((len(lens) * seg, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    layer.linear_segments(to_device(A, "bf16"), to_device(W, "bf16"), to_device(b, "bf16"),
                          torch.from_numpy(lens).cuda(), seg, out=C)
    torch.cuda.synchronize()
    ref = oracle.linear(A, W, b)
    got = to_host(C)
    for i, L in enumerate(lens):
        need = min((int(L) + 127) // 128 * 128, seg)
        rows = slice(i * seg, i * seg + need)
        assert_close(got[rows], ref[rows], "bf16", f"segment {i} (length {L})")


def test_linear_segments_edge_cases():
    """Every segment empty: no row block is needed, nothing is written (the kernel runs with
    no tiles).  Lengths past the segment count as the whole segment; segments shorter than
    one tile, and a row count that is not a multiple of 256, still give exact rows."""
    layer = Mha(64, 1, 64, dtype=torch.bfloat16)
    K, N = 128, 256
    W = wl.random_tensor((K, N), seed=32, scale=0.05)
    Wd = to_device(W, "bf16")
    for seg, lens in ((300, [0, 0, 0]), (300, [0, 301, 5]), (100, [3, 100, 0, 77, 50]),
                      (260, [260, 1, 130])):
        lens = np.array(lens, dtype=np.int32)
        A = wl.random_tensor((len(lens) * seg, K), seed=31)
        C = torch.full((len(lens) * seg, N), 7.0, dtype=torch.bfloat16, device="cuda")
        layer.linear_segments(to_device(A, "bf16"), Wd, None, torch.from_numpy(lens).cuda(), seg, out=C)
        torch.cuda.synchronize()
        got, ref = to_host(C), oracle.linear(A, W)
        if not lens.any():
            assert (got == 7.0).all()
        for i, L in enumerate(lens):
            need = min((min(max(int(L), 0), seg) + 127) // 128 * 128, seg)
            rows = slice(i * seg, i * seg + need)
            if need:
                assert_close(got[rows], ref[rows], "bf16", f"segment {i} of {seg} (length {L})")


def test_linear_strided_operands():
    """Row strides wider than the rows (a column block of W_qkv, as the
    cross-attention path uses)."""
    M, K, N, ld = 200, 128, 192, 576
    A = wl.random_tensor((M, K), seed=4)
    Wfull = wl.random_tensor((K, ld), seed=5, scale=0.05)
    layer = Mha(64, 1, 64, dtype=torch.bfloat16)
    Wd = to_device(Wfull, "bf16")
    out = torch.zeros((M, ld), dtype=torch.bfloat16, device="cuda")
    layer.linear(to_device(A, "bf16"), Wd[:, 192:384], None, out=out[:, 64:256])
    torch.cuda.synchronize()
    ref = oracle.linear(A, Wfull[:, 192:384])
    assert_close(to_host(out[:, 64:256]), ref, "bf16", "strided linear")
    assert (to_host(out[:, :64]) == 0).all() and (to_host(out[:, 256:]) == 0).all()


# ------------------------------------------------------------------ step: fused attention

ATTN_CASES = [
    # B, T_q, T_kv, h, d, causal, lengths, scale
    (1, 128, 128, 1, 64, False, None, 1.0),
    (2, 200, 200, 3, 64, True, None, 1.0),
    (1, 129, 129, 2, 128, True, None, 1.0),
    (2, 127, 127, 2, 128, False, None, 1.0),
    (1, 1, 1, 2, 64, True, None, 1.0),                     # one query, one key
    (3, 70, 333, 2, 64, False, [1, 200, 333], 1.0),        # cross + padding incl. L=1, L=T_kv
    (2, 300, 300, 2, 64, True, [300, 129], 1.0),           # causal + padding
    (1, 384, 384, 2, 64, True, None, 4.0),                 # large scores: rescale path
    (2, 256, 520, 1, 128, False, [520, 257], 3.0),
    # more work items (query tile x (batch, head)) than the d = 64 kernel's persistent grid of
    # two CTAs per SM, so every CTA runs several items and starts item k+1 (its Q load, first K
    # tiles and first score MMA) while item k drains
    (8, 1024, 1024, 8, 64, True, None, 1.0),               # causal, 512 items
    (4, 1024, 1024, 16, 64, False, None, 1.0),             # no mask, 512 items
    (16, 384, 1000, 8, 64, False,                          # key lengths, batches sorted by
     [int(v) for v in np.random.default_rng(5).integers(1, 1001, 16)], 1.0),  # length, 384 items
]


@pytest.mark.parametrize("B,T_q,T_kv,h,d,causal,lengths,scale", ATTN_CASES)
def test_attention_step_bf16(B, T_q, T_kv, h, d, causal, lengths, scale):
    Q = wl.random_tensor((B, T_q, h * d), seed=10, scale=scale)
    K = wl.random_tensor((B, T_kv, h * d), seed=11, scale=scale)
    V = wl.random_tensor((B, T_kv, h * d), seed=12)
    kvl = None if lengths is None else np.array(lengths, dtype=np.int32)
    layer = Mha(h * d, h, d, dtype=torch.bfloat16)
    layer.ensure_workspace(1, 1, 1)
    O = layer.attention(to_device(Q, "bf16"), to_device(K, "bf16"), to_device(V, "bf16"),
                        causal=causal,
                        kv_lengths=None if kvl is None else torch.from_numpy(kvl).cuda())
    torch.cuda.synchronize()
    assert layer.status() == _lib.MHA_OK
    ref = oracle.attention(Q, K, V, h=h, causal=causal, kv_lengths=kvl)
    assert_close(to_host(O), ref, "bf16", f"attention {B}x{T_q}x{T_kv} h{h} d{d}")


@pytest.mark.parametrize("ramp_top", [12.0, 40.0])
@pytest.mark.parametrize("d,causal", [(64, True), (64, False), (128, True), (128, False)])
def test_attention_growing_scores_bf16(d, causal, ramp_top):
    """Scores that grow steeply along the keys: each key tile's maximum is far above the
    previous tiles'.  With the steeper ramp later tiles exceed the first tile's maximum by
    far more than 64 (in base-2 units), so the kernel must leave its no-maximum fast path,
    move its reference maximum and rescale O and the row sums."""
    B, T, h = 1, 640, 2
    Q = wl.random_tensor((B, T, h * d), seed=30, scale=1.0)
    Kb = wl.random_tensor((B, T, h * d), seed=31, scale=1.0)
    ramp = (0.2 + ramp_top * np.arange(T, dtype=np.float32) / T)[None, :, None]
    K = wl.round_to_bf16(Kb * ramp)
    V = wl.random_tensor((B, T, h * d), seed=32)
    layer = Mha(h * d, h, d, dtype=torch.bfloat16)
    layer.ensure_workspace(1, 1, 1)
    O = layer.attention(to_device(Q, "bf16"), to_device(K, "bf16"), to_device(V, "bf16"),
                        causal=causal)
    torch.cuda.synchronize()
    assert layer.status() == _lib.MHA_OK
    ref = oracle.attention(Q, K, V, h=h, causal=causal)
    assert_close(to_host(O), ref, "bf16", f"growing scores d{d} causal={causal}")


@pytest.mark.parametrize("B,T_q,T_kv,h,dk,dv,causal,lengths", [
    (1, 16, 16, 8, 4, 4, False, None),
    (2, 77, 77, 3, 16, 8, True, None),
    (2, 40, 90, 2, 64, 96, False, [1, 90]),
    (1, 33, 33, 1, 256, 256, True, None),
])
def test_attention_step_f32(B, T_q, T_kv, h, dk, dv, causal, lengths):
    Q = wl.random_tensor((B, T_q, h * dk), seed=20, dtype="f32")
    K = wl.random_tensor((B, T_kv, h * dk), seed=21, dtype="f32")
    V = wl.random_tensor((B, T_kv, h * dv), seed=22, dtype="f32")
    kvl = None if lengths is None else np.array(lengths, dtype=np.int32)
    layer = Mha(h * dk, h, dk, dv, dtype=torch.float32)
    O = layer.attention(to_device(Q, "f32"), to_device(K, "f32"), to_device(V, "f32"),
                        causal=causal,
                        kv_lengths=None if kvl is None else torch.from_numpy(kvl).cuda())
    torch.cuda.synchronize()
    ref = oracle.attention(Q, K, V, h=h, causal=causal, kv_lengths=kvl)
    assert_close(to_host(O), ref, "f32", "f32 attention")


# ------------------------------------------------------------------ whole forward, small

SMALL = [
    wl.custom("bf16_d64_causal", B=2, T_q=300, D=256, h=4, d_k=64, causal=True),
    wl.custom("bf16_d128_causal", B=1, T_q=260, D=512, h=4, d_k=128, causal=True),
    wl.custom("bf16_d64_full", B=3, T_q=129, D=192, h=3, d_k=64, causal=False, bias="none"),
    wl.custom("bf16_cross_pad", B=3, T_q=100, T_kv=333, D=256, h=4, d_k=64, cross=True,
              kv_len_range=(1, 333)),
    wl.custom("bf16_cross_d128", B=2, T_q=64, T_kv=200, D=256, h=2, d_k=128, cross=True,
              kv_len_range=(100, 200), bias="none"),
    wl.custom("f32_odd", B=2, T_q=37, D=48, h=3, d_k=16, d_v=8, dtype="f32", causal=True,
              weight_init="xavier_uniform", bias="uniform_0.1"),
    wl.custom("f32_cross", B=2, T_q=20, T_kv=45, D=64, h=4, d_k=16, dtype="f32", cross=True,
              kv_len_range=(1, 45), weight_init="uniform_inv_sqrt_d", bias="uniform_0.1"),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_forward_small(w):
    x = wl.make_inputs(w, seed=3)
    layer, y = _run_forward(w, x)
    assert layer.status() == _lib.MHA_OK
    assert_close(to_host(y), _oracle_forward(w, x), w.dtype, w.name)


# ------------------------------------------------------------------ named workloads, full size

@pytest.mark.parametrize("name", ["c1_f32_tiny", "c2_f32_causal"])
def test_named_f32_full(name):
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w)
    layer, y = _run_forward(w, x)
    assert layer.status() == _lib.MHA_OK
    e = assert_close(to_host(y), _oracle_forward(w, x), "f32", name)
    print(name, e)


@pytest.mark.parametrize("name", ["c3_bf16_causal", "c4_bf16_causal_long", "c5_bf16_cross"])
def test_named_bf16_full(name):
    """The full-size bf16 workloads through mha_forward (as the benchmark runs it), every
    output element against the oracle.  c3 runs 1024 work items on the persistent d = 64
    attention kernel (several per CTA), c5 768 with key lengths; c4 is one 16384-long causal
    sequence at d = 128 (the oracle needs about a minute of host time for it)."""
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w)
    layer, y = _run_forward(w, x)
    assert layer.status() == _lib.MHA_OK
    got = to_host(y)
    del y
    e = assert_close(got, _oracle_forward(w, x), "bf16", name)
    print(name, e)


# ------------------------------------------------------------------ edge cases

def test_invalid_lengths_give_nan_rows_and_status():
    """molayo1419.me pitfall 3: a sample whose keys are all excluded has an
    undefined softmax; its rows come out NaN and the call reports it."""
    for dtype in ("bf16", "f32"):
        w = wl.custom("badlen", B=3, T_q=50, T_kv=140, D=128, h=2, d_k=64, cross=True,
                      kv_len_range=(1, 140), dtype=dtype)
        x = wl.make_inputs(w, seed=5)
        x["kv_lengths"] = np.array([0, 77, 141], dtype=np.int32)
        layer, y = _run_forward(w, x)
        assert layer.status() == _lib.MHA_ERR_BAD_LENGTH
        assert layer.status() == _lib.MHA_OK  # reading clears it
        yh = to_host(y)
        assert np.isnan(yh[0]).all() and np.isnan(yh[2]).all()
        ref = _oracle_forward(w, {**x, "kv_lengths": np.array([1, 77, 1], dtype=np.int32)})
        assert_close(yh[1], ref[1], dtype, "valid batch next to invalid ones")


def test_padding_rows_do_not_matter_and_runs_are_deterministic():
    w = wl.custom("padinv", B=2, T_q=64, T_kv=300, D=256, h=4, d_k=64, cross=True,
                  kv_len_range=(130, 250))
    x = wl.make_inputs(w, seed=6)
    layer, y1 = _run_forward(w, x)
    _, y1b = _run_forward(w, x, layer)
    assert torch.equal(y1, y1b)
    x2 = dict(x)
    xkv = x["X_kv"].copy()
    for b, L in enumerate(x["kv_lengths"]):
        xkv[b, L:] = wl.round_to_bf16(np.full_like(xkv[b, L:], 30.0))
    x2["X_kv"] = xkv
    _, y2 = _run_forward(w, x2, layer)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("d", [64, 128])
def test_cross_projection_leaves_unread_key_rows_alone(d):
    """The key/value projection of cross-attention skips the 256-row blocks that lie past
    every batch's key length (in whole 128-key tiles).  The workspace starts as NaN, so a
    skipped row that the attention step did read would poison its batch's output.  T_kv is
    not a multiple of 256, so row blocks straddle batches; the lengths cover 1 key, one
    tile, a tile edge, and the whole sequence."""
    w = wl.custom(f"skiprows{d}", B=5, T_q=70, T_kv=700, D=256, h=256 // d, d_k=d, cross=True,
                  kv_len_range=(1, 700))
    x = wl.make_inputs(w, seed=12)
    x["kv_lengths"] = np.array([1, 127, 128, 300, 700], dtype=np.int32)
    layer = _layer(w)
    layer.ensure_workspace(w.B, w.T_q, w.T_kv).fill_(255)  # bf16 0xFFFF is a NaN
    layer.status()  # the fill also hit the status word: read it to clear it
    layer, y = _run_forward(w, x, layer)
    assert layer.status() == _lib.MHA_OK
    yh = to_host(y)
    assert np.isfinite(yh).all()
    assert_close(yh, _oracle_forward(w, x), "bf16", w.name)


ROUNDED_CASES = [
    wl.custom("rnd_causal64", B=2, T_q=300, D=256, h=4, d_k=64, causal=True),
    wl.custom("rnd_causal128", B=1, T_q=400, D=256, h=2, d_k=128, causal=True),
    wl.custom("rnd_cross64", B=3, T_q=100, T_kv=500, D=256, h=4, d_k=64, cross=True,
              kv_len_range=(1, 500)),
]


@pytest.mark.parametrize("w", ROUNDED_CASES, ids=[w.name for w in ROUNDED_CASES])
def test_bf16_path_tracks_the_rounded_oracle(w):
    """Secondary diagnostic: the oracle's rounded mode stores Q/K/V, the softmax weights, the
    attention output and Y as bf16 where the GPU path does.  The GPU result must sit closer to
    it than to the unrounded oracle, and nearly every output within one bf16 unit in the last
    place of it.  What remains is not rounding placement: the GPU rounds each softmax weight
    against a different reference maximum (an independent rounding of the same size), sums in
    fp32, and any such difference upstream flips some final roundings by one unit."""
    x = wl.make_inputs(w, seed=14)
    layer, y = _run_forward(w, x)
    got = to_host(y)
    plain = _oracle_forward(w, x)
    rounded = oracle.mha_forward(x["X_q"], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h, w.d_k,
                                 w.d_v, Xkv=x["X_kv"], causal=w.causal, kv_lengths=x["kv_lengths"],
                                 round_bf16=True)
    e_plain = np.linalg.norm(got - plain) / np.linalg.norm(plain)
    e_round = np.linalg.norm(got - rounded) / np.linalg.norm(rounded)
    # distance in bf16 units in the last place of the rounded value (8 significant bits;
    # values below 1% of the rms count as that size, where a ulp is meaningless)
    floor = 0.01 * np.sqrt(np.mean(rounded ** 2))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rounded), floor))) - 7)
    d_ulp = np.abs(got - rounded) / ulp
    print(w.name, "rel Frobenius vs plain", e_plain, "vs rounded", e_round,
          "ulps: max", d_ulp.max(), "p99.9", np.quantile(d_ulp, 0.999), "share > 1", np.mean(d_ulp > 1))
    assert e_round <= 0.7 * e_plain, (e_round, e_plain)
    assert np.mean(d_ulp > 1) <= 0.1


def test_forward_checked_matches_forward_and_rejects_bad_lengths():
    w = wl.custom("checked", B=3, T_q=40, T_kv=300, D=256, h=4, d_k=64, cross=True,
                  kv_len_range=(1, 300))
    x = wl.make_inputs(w, seed=13)
    layer, y = _run_forward(w, x)
    d = {k: to_device(v, w.dtype) for k, v in x.items() if k != "kv_lengths"}
    kvl = torch.from_numpy(x["kv_lengths"]).cuda()
    y2 = torch.empty_like(y)
    stream = torch.cuda.current_stream().cuda_stream
    args = (layer.handle, d["X_q"].data_ptr(), d["X_kv"].data_ptr(), w.B, w.T_q, w.T_kv,
            d["W_qkv"].data_ptr(), d["b_qkv"].data_ptr(), d["W_o"].data_ptr(), d["b_o"].data_ptr(), 0,
            kvl.data_ptr())
    assert _lib.mha_forward_checked(*args, x["kv_lengths"], y2.data_ptr(), stream) == _lib.MHA_OK
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    bad = x["kv_lengths"].copy()
    bad[1] = 0
    y3 = torch.full_like(y, 7.0)
    code = _lib.mha_forward_checked(*args, bad, y3.data_ptr(), stream, check=False)
    torch.cuda.synchronize()
    assert code == _lib.MHA_ERR_BAD_LENGTH
    assert (y3 == 7.0).all()  # nothing was launched
    assert layer.status() == _lib.MHA_OK


def test_output_guard_bands_untouched():
    w = wl.custom("guard", B=2, T_q=131, D=256, h=4, d_k=64, causal=True)
    x = wl.make_inputs(w, seed=7)
    layer = _layer(w)
    d = {k: to_device(v, w.dtype) for k, v in x.items() if k != "kv_lengths"}
    n = w.B * w.T_q * w.D
    pad = 4096
    buf = torch.full((n + 2 * pad,), 12345.0, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + n].view(w.B, w.T_q, w.D)
    layer.forward(d["X_q"], d["W_qkv"], d["b_qkv"], d["W_o"], d["b_o"], causal=True, out=out)
    torch.cuda.synchronize()
    assert (buf[:pad] == 12345.0).all() and (buf[pad + n:] == 12345.0).all()
    assert_close(to_host(out), _oracle_forward(w, x), "bf16", "guard")


def test_empty_batch_is_a_no_op():
    layer = Mha(256, 4, 64, dtype=torch.bfloat16)
    X = torch.empty((0, 10, 256), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 768), dtype=torch.bfloat16, device="cuda")
    Wo = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    y = layer.forward(X, W, None, Wo, None)
    torch.cuda.synchronize()
    assert y.shape == (0, 10, 256)
