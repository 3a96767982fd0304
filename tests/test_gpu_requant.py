"""GPU parity of moe_mx_requant (BF16 -> MXFP8 -> BF16, the conventional
path's activation round trip) against the oracle, bit for bit, and the
accuracy comparison that the warp-decode page's accuracy section makes:
the BF16-activation path (moe_layer) against the conventional path's
numerics (x and h converted before their GEMMs), both measured against the
FP64 truth (x as given, h unrounded)."""
import json
import os

import numpy as np
import pytest
import torch

import mixture_experts_decode_gb300 as moe
import oracle
from mixture_experts_decode_gb300 import inputs

from _gpu_helpers import WEIGHT_NAMES, check_close, check_cosine, device_mx, run_layer

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def _bf16(vals: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(vals, dtype=np.float64)).to(torch.bfloat16)


def _inputs(kind: str, rows: int, K: int, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    if kind == "normal":
        v = rng.standard_normal((rows, K)) * 0.5
    elif kind == "wide":       # exponents over [-60, 60] inside one block
        v = np.ldexp(rng.uniform(0.5, 1.0, (rows, K)), rng.integers(-60, 60, (rows, K)))
        v *= rng.choice([-1.0, 1.0], (rows, K))
    elif kind == "ties":       # every value a midpoint of the E4M3 grid at the block exponent
        grid = sorted({oracle.e4m3_decode(c) for c in range(0, 0x7E)})
        mids = np.array([(a + b) / 2 for a, b in zip(grid, grid[1:])])
        X = rng.integers(-40, 40, (rows, K // 32))
        v = rng.choice(mids, (rows, K)) * rng.choice([-1.0, 1.0], (rows, K))
        v[:, ::32] = 448.0 * np.sign(v[:, ::32])          # pin each block's exponent
        v = v * np.repeat(np.ldexp(1.0, X), 32, axis=1)
    elif kind == "saturate":   # block maxima in (448, 512) * 2^X
        v = rng.uniform(-1, 1, (rows, K)) * 256.0
        v[:, ::32] = rng.uniform(449, 511, (rows, K // 32))
        v = v * np.ldexp(1.0, -8)
    elif kind == "zeros":
        v = np.zeros((rows, K))
        v[::2, 3::32] = -0.0
        v[1::3, 5] = 1.5
    elif kind == "tiny":       # BF16 subnormals and the E8M0 clamp
        v = np.ldexp(rng.uniform(-1, 1, (rows, K)), rng.integers(-133, -118, (rows, K)))
    else:
        raise ValueError(kind)
    return _bf16(v)


@pytest.mark.parametrize("kind", ["normal", "wide", "ties", "saturate", "zeros", "tiny"])
@pytest.mark.parametrize("rows,K", [(1, 32), (37, 96), (64, 2048)])
def test_requant_matches_oracle(cuda_device, kind, rows, K):
    x = _inputs(kind, rows, K, rows * 1000 + K)
    got = moe.mx_requant(x.to(cuda_device))
    torch.cuda.synchronize()
    want = oracle.mx_requant(_bits(x))
    g = _bits(got)
    bad = np.flatnonzero(g != want)
    assert bad.size == 0, f"{kind} {rows}x{K}: {bad.size} differ, first at {bad[:4]}: {g.flat[bad[:4]]} vs {want.flat[bad[:4]]}"


def test_requant_large_and_in_place(cuda_device):
    x = _inputs("normal", 4099, 2048, 5)          # ragged last CTA
    xd = x.to(cuda_device)
    out = moe.mx_requant(xd)
    moe.mx_requant(xd, out=xd)                    # in place
    torch.cuda.synchronize()
    want = oracle.mx_requant(_bits(x))
    np.testing.assert_array_equal(_bits(out), want)
    np.testing.assert_array_equal(_bits(xd), want)


def test_requant_leaves_neighbours_alone(cuda_device):
    x = _inputs("wide", 7, 64, 6).to(cuda_device)
    buf = torch.full((7 * 64 + 4096,), 1234.0, dtype=torch.bfloat16, device=cuda_device)
    view = buf[:7 * 64].view(7, 64)
    moe.mx_requant(x, out=view)
    torch.cuda.synchronize()
    assert bool((buf[7 * 64:] == 1234.0).all())
    np.testing.assert_array_equal(_bits(view), oracle.mx_requant(_bits(x.cpu())))


@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_requant_16_byte_aligned_buffers(cuda_device, kind):
    """Buffers 16- but not 32-byte aligned take the 16-byte (four threads per
    block) path; in place there too."""
    x = _inputs(kind, 19, 160, 7)
    n = x.numel()
    src = torch.zeros(n + 16, dtype=torch.bfloat16, device=cuda_device)
    dst = torch.full((n + 4096,), 1234.0, dtype=torch.bfloat16, device=cuda_device)
    xin = src[8:8 + n].view(19, 160)              # +16 bytes
    xin.copy_(x.to(cuda_device))
    out = dst[8:8 + n].view(19, 160)
    assert xin.data_ptr() % 32 == 16 and out.data_ptr() % 32 == 16
    moe.mx_requant(xin, out=out)
    torch.cuda.synchronize()
    want = oracle.mx_requant(_bits(x))
    np.testing.assert_array_equal(_bits(out), want)
    assert bool((dst[:8] == 1234.0).all()) and bool((dst[8 + n:] == 1234.0).all())
    moe.mx_requant(xin, out=xin)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(xin), want)


def test_requant_empty(cuda_device):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda_device)
    assert moe.mx_requant(x).shape == (0, 64)


# ------------------------------------------------- conventional path ---

def _conventional(dev, Wd, x, ids, w):
    """The conventional path's numerics through the C-ABI: x and h each go
    through moe_mx_requant before their pass."""
    xq = moe.mx_requant(x.to(dev))
    h = moe.gate_up(xq, ids.to(dev), Wd["gate"], Wd["up"])
    hq = moe.mx_requant(h)
    y = moe.down(hq, ids.to(dev), w.to(dev), Wd["down"])
    return h, y


def _oracle_subset(fn, W, x, ids, w, tokens, **kw):
    tokens = list(tokens)
    sub = ids[tokens].cpu().numpy()
    uniq = sorted(set(sub.reshape(-1).tolist()))
    remap = np.full(max(uniq) + 1, -1, np.int64)
    remap[uniq] = np.arange(len(uniq))
    idx = torch.tensor(uniq, dtype=torch.long)
    host = [W[n].index_select(0, idx.to(W[n].device)).cpu().numpy() for n in WEIGHT_NAMES]
    return fn(_bits(x[tokens]), remap[sub].astype(np.int32), w[tokens].cpu().numpy(), *host, **kw)


@pytest.fixture(scope="module")
def qwen(cuda_device):
    W = inputs.layer_weights(inputs.QWEN3, cuda_device)
    return W, device_mx(W, cuda_device)


def test_conventional_path_matches_oracle(cuda_device, qwen):
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, 4)
    h, y = _conventional(cuda_device, Wd, x, ids, w)
    torch.cuda.synchronize()
    ref = _oracle_subset(oracle.moe_layer_mx_act, W, x, ids, w, range(4))
    check_close(h, ref["h64"], "conventional h")
    check_close(y, ref["y64"], "conventional y")
    check_cosine(y, ref["y64"], "conventional y")


def test_bf16_path_is_closer_to_the_fp64_truth(cuda_device, qwen):
    """At the B=32 workload: per token, the relative L2 distance of y to the
    FP64 truth for moe_layer (BF16 activations) and for the conventional
    path; the BF16 path must be the closer one for every token.  The
    measured distances go to $MOE_ACCURACY_OUT (JSON) when it is set."""
    W, Wd = qwen
    B = 32
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    y_wd = run_layer(cuda_device, Wd, x, ids, w)
    _, y_cv = _conventional(cuda_device, Wd, x, ids, w)
    torch.cuda.synchronize()
    toks = [0, 5, 11, 17, 23, 31]
    t = _oracle_subset(oracle.moe_layer, W, x, ids, w, toks, want_truth=True)["truth64"]
    idx = torch.tensor(toks, device=cuda_device)
    e = {}
    for name, y in (("bf16_path", y_wd), ("conventional", y_cv)):
        yy = y.index_select(0, idx).double().cpu().numpy()
        e[name] = np.linalg.norm(yy - t, axis=1) / np.linalg.norm(t, axis=1)
    assert np.all(e["conventional"] > e["bf16_path"]), e
    res = {"workload": "qwen3_e128_k8_d2048_i768 B=32", "tokens": toks,
           "rel_l2_bf16_path": e["bf16_path"].tolist(), "rel_l2_conventional": e["conventional"].tolist(),
           "mean_ratio": float(np.mean(e["conventional"]) / np.mean(e["bf16_path"]))}
    out = os.environ.get("MOE_ACCURACY_OUT")
    if out:
        with open(out, "w") as f:
            json.dump(res, f, indent=1)
