"""Pins for the CPU oracle: each test ties it to something other than itself.

Sources: MXFP8 code tables (OCP OFP8 / MX v1.0, the format "Warp decode"
names for its weights), library routines (torch float8 casts, numpy float64
matmuls), closed forms and invariants of the decode layer ("Warp decode",
how the two kernels work), and brute force for MoE Align & Sort.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_decode_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((a, b))
    return rows


# ------------------------------------------------------------ MX codes ---

def test_e4m3_golden_codes():
    for code, val in _table("e4m3_codes.txt"):
        got = oracle.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val), (code, got, val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val)), code


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_e4m3_monotone_and_symmetric():
    pos = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    for c in range(0x7F):
        assert oracle.e4m3_decode(c | 0x80) == -pos[c]


def test_e8m0_golden_codes():
    for code, p in _table("e8m0_codes.txt"):
        got = oracle.e8m0_decode(int(code))
        if p == "nan":
            assert math.isnan(got)
        else:
            assert got == math.ldexp(1.0, int(p))


def test_e8m0_matches_torch_when_available():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch has no float8_e8m0fnu")
    codes = torch.arange(255, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float32).double().numpy()
    for c in range(255):
        assert oracle.e8m0_decode(c) == ref[c], c


# ---------------------------------------------------------------- BF16 ---

def _bf16_value(bits):
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def test_bf16_round_is_nearest_ties_even_brute_force():
    rng = random.Random(1234)
    for _ in range(4000):
        v = rng.uniform(-1, 1) * math.ldexp(1.0, rng.randint(-140, 127))
        b = oracle.bf16_round(v)
        r = _bf16_value(b)
        # neighbours of the result in bf16 bit space must not be closer
        for nb in ((b + 1) & 0xFFFF, (b - 1) & 0xFFFF):
            rv = _bf16_value(nb)
            if math.isfinite(rv) and (rv == 0 or math.copysign(1, rv) == math.copysign(1, r)):
                assert abs(v - r) <= abs(v - rv), (v, r, rv)
                if abs(v - r) == abs(v - rv):
                    assert (b & 1) == 0, "tie must go to the even pattern"


def test_bf16_round_exact_midpoints_go_to_even():
    one = 1.0
    ulp = math.ldexp(1.0, -7)
    assert oracle.bf16_round(one + ulp / 2) == 0x3F80          # tie -> even (1.0)
    assert oracle.bf16_round(one + 3 * ulp / 2) == 0x3F82      # tie -> even (1 + 2 ulp)
    assert oracle.bf16_round(one + ulp / 2 + 1e-12) == 0x3F81  # above tie -> up
    assert oracle.bf16_round(-(one + ulp / 2)) == 0xBF80
    assert oracle.bf16_round(3.5e38) == 0x7F80                 # overflow -> inf
    assert oracle.bf16_round(math.ldexp(1.0, -133)) == 0x0001  # smallest subnormal
    assert oracle.bf16_round(math.ldexp(1.0, -134)) == 0x0000  # tie with 0 -> even (0)


def test_bf16_round_matches_torch_on_float32_inputs():
    g = torch.Generator().manual_seed(7)
    v = torch.randn(5000, generator=g, dtype=torch.float32) * torch.exp2(
        torch.randint(-30, 30, (5000,), generator=g).float())
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    for x, r in zip(v.double().tolist(), ref.tolist()):
        assert oracle.bf16_round(x) == r


# ------------------------------------------------------ MX quantiser ---

def _dequant_np(codes, scales):
    """Library dequant: torch float8 cast, times 2^(s-127) via ldexp."""
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.repeat(scales.astype(np.int64) - 127, 32, axis=-1)
    return np.ldexp(c, s)


def test_quantizer_round_trips_representable_blocks():
    rng = np.random.default_rng(3)
    reps = []
    for X in (-20, -7, 0, 5):
        q = rng.integers(0, 256, size=32).astype(np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x38          # no NaNs
        q[0] = 0x7E                            # amax = 448 * 2^X -> X recovered
        vals = np.array([oracle.e4m3_decode(int(c)) for c in q]) * 2.0 ** X
        reps.append((vals, q, X))
    v = torch.tensor(np.stack([r[0] for r in reps]), dtype=torch.float32)
    codes, scales = inputs.quantize_mx(v)
    for i, (vals, q, X) in enumerate(reps):
        assert int(scales[i, 0]) == X + 127
        back = np.array([oracle.e4m3_decode(int(c)) for c in codes[i].numpy()]) * 2.0 ** X
        np.testing.assert_array_equal(back, vals)


def test_quantizer_zero_block_and_range():
    v = torch.zeros((2, 64))
    v[1] = torch.randn(64, generator=torch.Generator().manual_seed(11)) * 0.02
    codes, scales = inputs.quantize_mx(v)
    assert int(scales[0, 0]) == 127 and int(scales[0, 1]) == 127
    assert int(codes[0].abs().sum()) == 0
    deq = _dequant_np(codes.numpy(), scales.numpy())
    # X = floor(log2 amax) - 8 puts each block's largest |v| / 2^X in [256, 512);
    # values above 448 saturate to 448, the rest round to nearest (at most
    # half an ulp of the top E4M3 binade, 16 * 2^X)
    for blk in range(2):
        x = v[1, blk * 32:(blk + 1) * 32].double().numpy()
        q = deq[1, blk * 32:(blk + 1) * 32]
        X = int(scales[1, blk]) - 127
        assert 256 <= np.max(np.abs(x)) / 2.0 ** X < 512
        sat = np.abs(x) > 448 * 2.0 ** X
        assert np.all(np.abs(q[sat]) == 448 * 2.0 ** X)
        assert np.all(np.abs(q[~sat] - x[~sat]) <= 16 * 2.0 ** X)


def test_quantizer_saturates_top_binade():
    v = torch.zeros((1, 32))
    v[0, 0] = 500.0                    # X = 0: 500 > 448 saturates
    v[0, 1] = -300.0
    codes, scales = inputs.quantize_mx(v)
    assert int(scales[0, 0]) == 127
    assert oracle.e4m3_decode(int(codes[0, 0])) == 448.0
    assert oracle.e4m3_decode(int(codes[0, 1])) == -288.0   # nearest E4M3 (ulp 32), ties even


# ---------------------------------------------------------- FFN layer ---

def _mk(E, I, d, seed, shared=False):
    dev = "cpu"
    wg, sg = inputs.mx_weights(E, I, d, dev, "pin", seed, "g")
    wu, su = inputs.mx_weights(E, I, d, dev, "pin", seed, "u")
    wd, sd = inputs.mx_weights(E, d, I, dev, "pin", seed, "d")
    W = [t.numpy() for t in (wg, sg, wu, su, wd, sd)]
    sh = None
    if shared:
        a = inputs.mx_weights(1, I, d, dev, "pin", seed, "sg")
        b = inputs.mx_weights(1, I, d, dev, "pin", seed, "su")
        c = inputs.mx_weights(1, d, I, dev, "pin", seed, "sd")
        sh = tuple(t.numpy() for t in (*a, *b, *c))
    return W, sh


def _x(B, d, seed):
    x = inputs.randn((B, d), "cpu", "pin-x", seed).to(torch.bfloat16)
    return x.view(torch.int16).numpy().astype(np.uint16), x.double().numpy()


def _dense_swiglu(xf, wg, sg, wu, su, wd, sd):
    """Textbook dense SwiGLU FFN with numpy float64 matmuls (unrounded h)."""
    Wg, Wu, Wd = _dequant_np(wg, sg), _dequant_np(wu, su), _dequant_np(wd, sd)
    g = xf @ Wg.T
    u = xf @ Wu.T
    h = g / (1.0 + np.exp(-g)) * u
    return h, h @ Wd.T


def test_k1_weight1_reduces_to_dense_swiglu():
    E, I, d, B = 3, 64, 96, 4
    W, _ = _mk(E, I, d, 11)
    xb, xf = _x(B, d, 11)
    ids = np.array([[2], [0], [1], [2]], dtype=np.int32)
    w = np.ones((B, 1), dtype=np.float32)
    out = oracle.moe_layer(xb, ids, w, *W, want_truth=True)
    for b in range(B):
        e = ids[b, 0]
        h, y = _dense_swiglu(xf[b:b + 1], *(a[e] for a in W))
        np.testing.assert_allclose(out["truth64"][b], y[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out["g64"][b, 0], xf[b] @ _dequant_np(W[0][e], W[1][e]).T,
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out["u64"][b, 0], xf[b] @ _dequant_np(W[2][e], W[3][e]).T,
                                   rtol=1e-12, atol=1e-12)
        # BF16 intermediate: within half a bf16 ulp of the exact value
        hb = torch.from_numpy(out["h"][b, 0].astype(np.int16)).view(torch.bfloat16).double().numpy()
        assert np.all(np.abs(hb - h[0]) <= np.abs(h[0]) * 2.0 ** -8 + 1e-300)
        # down pass applied to the oracle's own BF16 h
        Wd = _dequant_np(W[4][e], W[5][e])
        np.testing.assert_allclose(out["y64"][b], Wd @ hb, rtol=1e-12, atol=1e-12)


def test_permuting_topk_order_leaves_output_unchanged():
    E, I, d, B, k = 6, 32, 64, 3, 4
    W, _ = _mk(E, I, d, 5)
    xb, _ = _x(B, d, 5)
    ids, w = inputs.route("softmax_normal", B, E, k, "perm")
    ids, w = ids.numpy(), w.numpy()
    a = oracle.moe_layer(xb, ids, w, *W)["y64"]
    perm = np.array([2, 0, 3, 1])
    b = oracle.moe_layer(xb, ids[:, perm], w[:, perm], *W)["y64"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_zero_weights_and_zero_input_give_zero():
    E, I, d, B, k = 4, 32, 64, 2, 2
    W, _ = _mk(E, I, d, 6)
    xb, _ = _x(B, d, 6)
    ids, w = inputs.route("softmax_normal", B, E, k, "zero")
    Z = [np.zeros_like(a) if i % 2 == 0 else a for i, a in enumerate(W)]   # all codes 0
    assert np.all(oracle.moe_layer(xb, ids.numpy(), w.numpy(), *Z)["y64"] == 0.0)
    assert np.all(oracle.moe_layer(np.zeros_like(xb), ids.numpy(), w.numpy(), *W)["y64"] == 0.0)


def test_linear_in_routing_weights_and_duplicates_add():
    E, I, d, B = 5, 32, 64, 2
    W, _ = _mk(E, I, d, 8)
    xb, _ = _x(B, d, 8)
    ids = np.array([[1, 3], [4, 0]], dtype=np.int32)
    w = np.array([[0.25, 0.5], [0.125, 1.0]], dtype=np.float32)
    y = oracle.moe_layer(xb, ids, w, *W)["y64"]
    y3 = oracle.moe_layer(xb, ids, 3 * w, *W)["y64"]
    np.testing.assert_allclose(y3, 3 * y, rtol=1e-12, atol=1e-15)
    dup = oracle.moe_layer(xb, np.array([[2, 2], [2, 2]], np.int32),
                           np.array([[0.25, 0.5], [0.5, 0.25]], np.float32), *W)["y64"]
    one = oracle.moe_layer(xb, np.array([[2], [2]], np.int32),
                           np.array([[0.75], [0.75]], np.float32), *W)["y64"]
    np.testing.assert_allclose(dup, one, rtol=1e-12, atol=1e-15)


def test_shared_expert_alone_is_dense_ffn():
    E, I, d, B, k = 4, 32, 64, 2, 2
    W, sh = _mk(E, I, d, 9, shared=True)
    xb, xf = _x(B, d, 9)
    ids, _ = inputs.route("softmax_normal", B, E, k, "sh")
    w0 = np.zeros((B, k), np.float32)
    out = oracle.moe_layer(xb, ids.numpy(), w0, *W, shared=sh, want_truth=True)
    _, y = _dense_swiglu(xf, *(a[0] for a in sh))
    np.testing.assert_allclose(out["truth64"], y, rtol=1e-12, atol=1e-12)
    assert out["h"].shape == (B, k + 1, I)


def test_oracle_rejects_out_of_range_ids():
    W, _ = _mk(2, 32, 32, 1)
    xb, _ = _x(1, 32, 1)
    with pytest.raises(ValueError):
        oracle.moe_layer(xb, np.array([[2]], np.int32), np.ones((1, 1), np.float32), *W)


# -------------------------------------------------------------- align ---

def _brute_align(ids, E, bs):
    T, k = ids.shape
    N = T * k
    flat = ids.reshape(-1).tolist()
    order = sorted(range(N), key=lambda f: (flat[f], f))
    out, eids = [], []
    for e in range(E):
        run = [f for f in order if flat[f] == e]
        if not run:
            continue
        padded = run + [N] * ((-len(run)) % bs)
        out += padded
        eids += [e] * (len(padded) // bs)
    ntpp = len(out)
    n_sorted = N + E * (bs - 1)
    n_blocks = -(-n_sorted // bs)
    out += [N] * (n_sorted - len(out))
    eids += [-1] * (n_blocks - len(eids))
    return np.array(out, np.int32), np.array(eids, np.int32), ntpp


def test_align_golden_cases():
    with open(os.path.join(GOLDEN, "align_tiny.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        s, e, n = oracle.align(np.array(c["topk_ids"], np.int32), c["E"], c["block_size"])
        assert s.tolist() == c["sorted_token_ids"]
        assert e.tolist() == c["expert_ids"]
        assert n == c["num_tokens_post_pad"]


@pytest.mark.parametrize("T,k,E,bs", [(0, 2, 4, 4), (1, 1, 1, 1), (5, 3, 7, 2), (17, 4, 9, 8),
                                      (33, 8, 16, 16), (64, 2, 3, 5), (9, 8, 8, 64)])
def test_align_matches_brute_force(T, k, E, bs):
    rng = np.random.default_rng(T * 1000 + E)
    for trial in range(3):
        if trial == 2:
            ids = np.full((T, k), E - 1, np.int32)         # one hot expert
        else:
            ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        s, e, n = oracle.align(ids, E, bs)
        bs_, be, bn = _brute_align(ids, E, bs)
        assert n == bn
        np.testing.assert_array_equal(s, bs_)
        np.testing.assert_array_equal(e, be)


def test_align_closed_form_and_properties():
    ids = inputs.align_ids(256, 8, 32, "zipf")
    T, k = ids.shape
    E, bs = 32, 16
    s, e, n = oracle.align(ids.numpy(), E, bs)
    cnt = np.bincount(ids.numpy().reshape(-1), minlength=E)
    assert n == int(np.sum((cnt + bs - 1) // bs * bs))
    N = T * k
    real = s[s < N]
    assert sorted(real.tolist()) == list(range(N))         # each flat index exactly once
    flat = ids.numpy().reshape(-1)
    for blk in range(n // bs):
        members = s[blk * bs:(blk + 1) * bs]
        members = members[members < N]
        assert np.all(flat[members] == e[blk])             # blocks are expert-homogeneous
        assert np.all(np.diff(members) > 0)                # stable: increasing flat index
    assert np.all(s[n:] == N) and np.all(e[n // bs:] == -1)
