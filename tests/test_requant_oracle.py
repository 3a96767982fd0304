"""Pins for the oracle's MXFP8 activation round trip (BF16 -> MXFP8 -> BF16)
and for the conventional-path layer built on it.

The round trip is the conventional expert-centric path's activation
conversion ("Warp decode", section "準確度改進"); the conversion rule is
OCP MX v1.0's (shared exponent floor(log2 max|v|) - 8 per 32 values, E4M3
elements nearest with ties to even, saturating at 448).  The pins: values
worked by hand from that rule, brute force over all finite E4M3 values,
torch's float8_e4m3fn cast (a library routine) through the seeded weight
quantiser, and invariants of the rule.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_decode_gb300 import inputs


def _bits(vals):
    t = torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def _vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _block(vals):
    v = list(vals) + [0.0] * (32 - len(vals))
    return np.array(v, dtype=np.float64)


# every finite E4M3 value with its code (the code tables are pinned elsewhere)
_E4M3 = sorted((oracle.e4m3_decode(c), c) for c in range(256) if not math.isnan(oracle.e4m3_decode(c)))


def _e4m3_brute(q):
    """Nearest finite E4M3 value by exhaustive search; ties to the even code;
    beyond 448 the largest finite value."""
    if abs(q) > 448.0:
        return math.copysign(448.0, q)
    best = None
    for v, c in _E4M3:
        dist = abs(v - q)
        if best is None or dist < best[0] or (dist == best[0] and (c & 1) == 0 and (best[2] & 1) == 1):
            best = (dist, v, c)
    v = best[1]
    return math.copysign(abs(v), q) if v == 0.0 else v


# ---------------------------------------------------------- hand-worked ---

def test_hand_worked_block():
    # amax 1.75 -> X = floor(log2 1.75) - 8 = -8; v * 256 on the E4M3 grid
    # (spacing 32 in [256, 512), 2 in [16, 32), 2^-9 below 2^-6)
    vals = [1.0, 1.0 + 2 ** -7, 1.0625, 1.1875, 1.75, 0.0625, -1.0625, 0.0,
            2 ** -14, 3 * 2 ** -18, 2 ** -18]
    want = [1.0, 1.0, 1.0, 1.25, 1.75, 0.0625, -1.0, 0.0,
            2 ** -14, 2 ** -16, 0.0]
    got = _vals(oracle.mx_requant(_bits(_block(vals)).reshape(1, 32)))[0]
    np.testing.assert_array_equal(got[:len(want)], want)
    assert np.all(got[len(want):] == 0)


def test_hand_worked_saturation_and_scale():
    # amax 1.9375: 1.9375 * 256 = 496 > 448 saturates to 1.75
    got = _vals(oracle.mx_requant(_bits(_block([1.9375, 1.0, -1.9375])).reshape(1, 32)))[0]
    assert list(got[:3]) == [1.75, 1.0, -1.75]
    # amax 300 -> X = 0: 300 -> 288 (spacing 32), 1.0 stays
    got = _vals(oracle.mx_requant(_bits(_block([300.0, 1.0, 17.0])).reshape(1, 32)))[0]
    assert list(got[:3]) == [288.0, 1.0, 16.0]   # 17 / 2 = 8.5 -> 8 (even)


def test_hand_worked_scale_clamp():
    # amax 2^-125 -> X = -133 clamps to -127; v * 2^127 stays on the grid
    vals = [2.0 ** -125, 3 * 2.0 ** -133]
    got = _vals(oracle.mx_requant(_bits(_block(vals)).reshape(1, 32)))[0]
    assert got[0] == 2.0 ** -125 and got[1] == 3 * 2.0 ** -133


def test_rejects_bad_block_length():
    with pytest.raises(ValueError):
        oracle.mx_requant(np.zeros((2, 48), dtype=np.uint16))


# ---------------------------------------------------------- brute force ---

def test_e4m3_round_matches_exhaustive_search():
    rng = np.random.default_rng(7)
    qs = list(rng.uniform(-600, 600, 3000)) + list(np.ldexp(rng.uniform(-1, 1, 3000), rng.integers(-12, 9, 3000)))
    # exact midpoints between neighbours, and the saturation edge
    for (a, _), (b, _) in zip(_E4M3, _E4M3[1:]):
        qs.append((a + b) / 2)
    qs += [448.0, 464.0, 479.9, 480.0, 1e6, -464.0, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11]
    for q in qs:
        assert oracle.e4m3_round(q) == _e4m3_brute(q), q


def test_round_trip_matches_brute_force():
    rng = np.random.default_rng(8)
    rows = []
    for r in range(12):
        mag = np.ldexp(rng.uniform(0.5, 1.0, 32), rng.integers(-30 + 4 * r, -20 + 4 * r, 32))
        rows.append(mag * rng.choice([-1.0, 1.0], 32))
    x_bits = _bits(np.array(rows))
    x = _vals(x_bits)
    got = _vals(oracle.mx_requant(x_bits))
    for i in range(len(rows)):
        amax = np.max(np.abs(x[i]))
        X = max(-127, min(127, math.frexp(amax)[1] - 1 - 8))
        want = [_e4m3_brute(math.ldexp(v, -X)) * 2.0 ** X for v in x[i]]
        want = torch.tensor(want, dtype=torch.float64).to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(got[i], want)


def test_round_trip_matches_torch_float8_quantiser():
    """The seeded weight quantiser converts float32 blocks with torch's
    float8_e4m3fn cast under the same OCP rule; dequantised and rounded to
    BF16 it must equal the oracle's round trip."""
    gen = torch.Generator().manual_seed(9)
    x = (torch.randn((64, 256), generator=gen) * torch.exp2(torch.randint(-20, 20, (64, 1), generator=gen).float()))
    xb = x.to(torch.bfloat16)
    codes, scales = inputs.quantize_mx(xb.float())
    c = codes.view(torch.float8_e4m3fn).double()
    s = torch.exp2(scales.double() - 127).repeat_interleave(32, dim=-1)
    want = (c * s).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = oracle.mx_requant(xb.view(torch.int16).numpy().astype(np.uint16))
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------- invariants ---

def test_invariants():
    gen = torch.Generator().manual_seed(10)
    x = (torch.randn((16, 128), generator=gen) * 3).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().astype(np.uint16)
    q = oracle.mx_requant(xb)
    # idempotent: a converted block keeps its shared exponent and its values
    np.testing.assert_array_equal(oracle.mx_requant(q), q)
    # odd: requant(-x) = -requant(x)
    neg = (-x).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(_vals(oracle.mx_requant(neg)), -_vals(q))
    # scaling by a power of two commutes (no clamp reached)
    for k in (-9, 5, 40):
        xs = (x.double() * 2.0 ** k).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
        np.testing.assert_array_equal(_vals(oracle.mx_requant(xs)), _vals(q) * 2.0 ** k)
    # each output block / 2^X is a set of E4M3 values
    finite = {v for v, _ in _E4M3}
    xv, qv = _vals(xb), _vals(q)
    for r in range(16):
        for b0 in range(0, 128, 32):
            X = math.frexp(np.max(np.abs(xv[r, b0:b0 + 32])))[1] - 1 - 8
            assert all(math.ldexp(v, -X) in finite for v in qv[r, b0:b0 + 32])


def test_zero_blocks_keep_their_bits():
    z = np.zeros((2, 64), dtype=np.uint16)
    z[1, 5] = 0x8000    # -0.0
    np.testing.assert_array_equal(oracle.mx_requant(z), z)


# --------------------------------------------- conventional-path layer ---

def _tiny_layer(B, seed):
    cfg = inputs.TINY
    W = inputs.layer_weights(cfg, "cpu")
    x, ids, w = inputs.layer_batch(cfg, B, step=seed)
    xb = x.view(torch.int16).numpy().astype(np.uint16)
    args = (xb, ids.numpy(), w.numpy(), *(W[n].numpy() for n in
                                          ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")))
    return args


def test_mx_act_gate_up_sees_converted_x():
    args = _tiny_layer(5, 0)
    conv = oracle.moe_layer_mx_act(*args)
    plain_on_qx = oracle.moe_layer(oracle.mx_requant(args[0]), *args[1:])
    np.testing.assert_array_equal(conv["h"], plain_on_qx["h"])
    np.testing.assert_array_equal(conv["h64"], plain_on_qx["h64"])


def test_mx_act_down_sees_converted_h():
    """y of the conventional path = the down projection of the converted
    BF16 h, written out here with numpy float64 matmuls."""
    args = _tiny_layer(3, 1)
    conv = oracle.moe_layer_mx_act(*args)
    ids, w = args[1], args[2]
    wd, sd = args[7], args[8]
    Wd = torch.from_numpy(wd).view(torch.float8_e4m3fn).double().numpy() * \
        np.repeat(np.ldexp(1.0, sd.astype(np.int64) - 127), 32, axis=-1)
    hq = _vals(oracle.mx_requant(conv["h"]))
    y = np.zeros_like(conv["y64"])
    for b in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            y[b] += float(w[b, j]) * (Wd[ids[b, j]] @ hq[b, j])
    np.testing.assert_allclose(conv["y64"], y, rtol=1e-12, atol=1e-15)


def test_conventional_path_is_farther_from_truth():
    """The BF16 path's y stays closer to the FP64 truth (h unrounded, x as
    given) than the conventional path's, token by token."""
    args = _tiny_layer(8, 2)
    plain = oracle.moe_layer(*args, want_truth=True)
    conv = oracle.moe_layer_mx_act(*args)
    t = plain["truth64"]
    e_plain = np.linalg.norm(plain["y64"] - t, axis=1)
    e_conv = np.linalg.norm(conv["y64"] - t, axis=1)
    assert np.all(e_conv > e_plain)
