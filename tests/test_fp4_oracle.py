"""Pins for the oracle's MXFP4-weight layer (the FP4 variant: E2M1 codes,
two per byte with the lower K index in the low nibble, one E8M0 scale per 32
along K; OCP MX v1.0) and for the seeded MXFP4 weight quantiser.

Sources: the OCP MX v1.0 E2M1 code table (tests/golden/e2m1_codes.txt), a
dense numpy float64 SwiGLU FFN (k = 1, weight 1), and the MXFP8 oracle on
the same weights re-encoded exactly as E4M3 (every E2M1 value is an E4M3
value, so both formats describe the same real matrices).
"""
import math
import os

import numpy as np
import torch

import oracle
from mixture_experts_decode_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    out = {}
    with open(os.path.join(GOLDEN, "e2m1_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                out[int(c, 16)] = float(v)
    return out


E2M1 = _e2m1_table()


def _unpack(codes: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] E2M1 codes (low nibble = lower K index)."""
    lo, hi = codes & 15, codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)


def _dequant4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    vals = np.vectorize(E2M1.get)(_unpack(codes)).astype(np.float64)
    return np.ldexp(vals, np.repeat(scales.astype(np.int64) - 127, 32, axis=-1))


def test_e2m1_golden_codes():
    assert len(E2M1) == 16
    for c, v in E2M1.items():
        got = oracle.e2m1_decode(c)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), hex(c)


def test_quantizer_ties_saturation_and_nibble_order():
    # X = floor(log2 7) - 2 = 0: midpoints tie to the even code; 7 saturates to 6
    v = torch.tensor([[0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, -0.75, -0.2, 0.0] + [0.0] * 20])
    codes, scales = inputs.quantize_mx4(v)
    assert int(scales[0, 0]) == 127
    got = _unpack(codes.numpy())[0, :12]
    assert list(got) == [0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x7, 0x7, 0xA, 0x0, 0x0]


def test_quantizer_round_trips_representable_blocks():
    rng = np.random.default_rng(4)
    for X in (-30, -3, 0, 9):
        c = rng.integers(0, 16, 64)
        c[0] = 0x7                                  # amax = 6 * 2^X -> X recovered
        c[32] = 0xF
        vals = np.array([E2M1[int(k)] for k in c]) * 2.0 ** X
        codes, scales = inputs.quantize_mx4(torch.tensor(vals, dtype=torch.float32).reshape(1, 64))
        assert list(scales[0].numpy()) == [X + 127, X + 127]
        np.testing.assert_array_equal(_dequant4(codes.numpy(), scales.numpy())[0], vals)


def _mk4(E, I, d, seed, shared=False):
    wg, sg = inputs.mx4_weights(E, I, d, "cpu", "pin4", seed, "g")
    wu, su = inputs.mx4_weights(E, I, d, "cpu", "pin4", seed, "u")
    wd, sd = inputs.mx4_weights(E, d, I, "cpu", "pin4", seed, "d")
    W = [t.numpy() for t in (wg, sg, wu, su, wd, sd)]
    sh = None
    if shared:
        a = inputs.mx4_weights(1, I, d, "cpu", "pin4", seed, "sg")
        b = inputs.mx4_weights(1, I, d, "cpu", "pin4", seed, "su")
        c = inputs.mx4_weights(1, d, I, "cpu", "pin4", seed, "sd")
        sh = tuple(t.numpy() for t in (*a, *b, *c))
    return W, sh


def _x(B, d, seed):
    x = inputs.randn((B, d), "cpu", "pin4-x", seed).to(torch.bfloat16)
    return x.view(torch.int16).numpy().astype(np.uint16), x.double().numpy()


def test_fp4_k1_weight1_reduces_to_dense_swiglu():
    E, I, d = 3, 64, 96
    W, _ = _mk4(E, I, d, 0)
    xb, xf = _x(4, d, 0)
    for e in range(E):
        ids = np.full((4, 1), e, dtype=np.int32)
        out = oracle.moe_layer(xb, ids, np.ones((4, 1), np.float32), *W, want_truth=True, fp4=True)
        Wg, Wu, Wd = _dequant4(W[0][e], W[1][e]), _dequant4(W[2][e], W[3][e]), _dequant4(W[4][e], W[5][e])
        g, u = xf @ Wg.T, xf @ Wu.T
        h = g / (1.0 + np.exp(-g)) * u
        np.testing.assert_allclose(out["g64"][:, 0], g, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["u64"][:, 0], u, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["truth64"], h @ Wd.T, rtol=1e-11, atol=1e-13)


def _as_mxfp8(codes4: np.ndarray) -> np.ndarray:
    """MXFP4 code bytes -> the same values as E4M3 codes (exact: every E2M1
    value is an E4M3 value), via torch's float8_e4m3fn cast."""
    vals = np.vectorize(E2M1.get)(_unpack(codes4)).astype(np.float32)
    return torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp4_layer_equals_mxfp8_layer_on_the_same_values():
    E, I, d, k, B = 6, 96, 128, 2, 5
    for shared in (False, True):
        W, sh = _mk4(E, I, d, 1 + shared, shared)
        xb, _ = _x(B, d, 1)
        rng = np.random.default_rng(3)
        ids = np.stack([rng.permutation(E)[:k] for _ in range(B)]).astype(np.int32)
        w = rng.random((B, k)).astype(np.float32)
        a = oracle.moe_layer(xb, ids, w, *W, shared=sh, want_truth=True, fp4=True)
        W8 = [_as_mxfp8(W[i]) if i % 2 == 0 else W[i] for i in range(6)]
        sh8 = None if sh is None else tuple(_as_mxfp8(sh[i]) if i % 2 == 0 else sh[i] for i in range(6))
        b = oracle.moe_layer(xb, ids, w, *W8, shared=sh8, want_truth=True)
        for key in ("h", "h64", "y64", "truth64"):
            np.testing.assert_array_equal(a[key], b[key], err_msg=f"{key} shared={shared}")
