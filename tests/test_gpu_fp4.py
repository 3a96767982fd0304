"""GPU parity of the MXFP4-weight passes (moe_gate_up_fp4, moe_down_fp4)
against the oracle's FP4 layer, through the C-ABI.  Tolerance as for the
MXFP8 layer: |gpu - oracle| <= 4e-3 * max(1, |oracle|) per element and
per-token cosine >= 0.99999 on y."""
import numpy as np
import pytest
import torch

import mixture_experts_decode_gb300 as moe
import oracle
from mixture_experts_decode_gb300 import inputs

from _gpu_helpers import WEIGHT_NAMES, check_close, check_cosine

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def _dev_weights(W, dev):
    mx = lambda a, b: moe.MX(W[a].to(dev), W[b].to(dev))
    out = dict(gate=mx("w_gate", "s_gate"), up=mx("w_up", "s_up"), down=mx("w_down", "s_down"), shared=None)
    if W.get("shared") is not None:
        s = [t.to(dev) for t in W["shared"]]
        out["shared"] = (moe.MX(s[0], s[1]), moe.MX(s[2], s[3]), moe.MX(s[4], s[5]))
    return out


def _run(dev, Wd, x, ids, w):
    sh = Wd["shared"]
    h = moe.gate_up(x.to(dev), ids.to(dev), Wd["gate"], Wd["up"], shared_gate=sh[0] if sh else None,
                    shared_up=sh[1] if sh else None, fp4=True)
    y = moe.down(h, ids.to(dev), w.to(dev), Wd["down"], shared_down=sh[2] if sh else None, fp4=True)
    torch.cuda.synchronize()
    return h, y


def _oracle(W, x, ids, w, tokens):
    """The FP4 oracle layer on `tokens`, passing only the experts they touch."""
    tokens = list(tokens)
    sub = ids[tokens].cpu().numpy()
    uniq = sorted(set(sub.reshape(-1).tolist()))
    remap = np.full(max(uniq) + 1, -1, np.int64)
    remap[uniq] = np.arange(len(uniq))
    idx = torch.tensor(uniq, dtype=torch.long)
    host = [W[n].index_select(0, idx.to(W[n].device)).cpu().numpy() for n in WEIGHT_NAMES]
    shared = None if W.get("shared") is None else tuple(t.cpu().numpy() for t in W["shared"])
    return oracle.moe_layer(_bits(x[tokens]), remap[sub].astype(np.int32), w[tokens].cpu().numpy(), *host,
                            shared=shared, fp4=True)


def _compare(dev, W, Wd, x, ids, w, tokens, what):
    h, y = _run(dev, Wd, x, ids, w)
    ref = _oracle(W, x, ids, w, tokens)
    t = torch.tensor(list(tokens), dtype=torch.long, device=dev)
    check_close(h.index_select(0, t), ref["h64"], what + " h")
    check_close(y.index_select(0, t), ref["y64"], what + " y")
    check_cosine(y.index_select(0, t), ref["y64"], what + " y")
    assert moe.device_error(dev) == 0


@pytest.mark.parametrize("B", [1, 3, 16])
def test_fp4_tiny_layer(cuda_device, B):
    W = inputs.layer_weights(inputs.TINY, "cpu", fp4=True)
    Wd = _dev_weights(W, cuda_device)
    x, ids, w = inputs.layer_batch(inputs.TINY, B)
    _compare(cuda_device, W, Wd, x, ids, w, range(B), f"fp4 tiny B={B}")


@pytest.fixture(scope="module")
def qwen4(cuda_device):
    W = inputs.layer_weights(inputs.QWEN3, cuda_device, fp4=True)
    return W, _dev_weights(W, cuda_device)


@pytest.mark.parametrize("B,routing", [(4, None), (8, None), (32, None), (32, "zipf")])
def test_fp4_qwen_layer_every_token(cuda_device, qwen4, B, routing):
    """The grouped MXFP4 kernels (every distinct expert's rows once per
    call, experts with more than four tokens in several groups)."""
    W, Wd = qwen4
    kw = {} if routing is None else {"routing": routing}
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B, **kw)
    _compare(cuda_device, W, Wd, x, ids, w, range(B), f"fp4 qwen B={B} {routing}")


def test_fp4_deepseek_shared_expert(cuda_device):
    """The grouped MXFP4 kernels with the always-on shared expert."""
    W = inputs.layer_weights(inputs.DEEPSEEK_V3, cuda_device, fp4=True)
    Wd = _dev_weights(W, cuda_device)
    x, ids, w = inputs.layer_batch(inputs.DEEPSEEK_V3, 8)
    _compare(cuda_device, W, Wd, x, ids, w, range(8), "fp4 deepseek B=8")
    del W, Wd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("E,k,d,I", [(4, 2, 512, 256), (3, 3, 1056, 64)])
def test_fp4_wide_scale_exponents(cuda_device, E, k, d, I):
    """Scale bytes spread over 127 +- 20 (weights from 2^-20 to 2^20 times
    their codes), on the grouped kernels (first shape) and the one-warp
    kernels (second): each block's scale must multiply exactly its own
    partial sum."""
    cfg = inputs.LayerConfig(f"fp4_wide_{E}_{k}_{d}_{I}", E, k, d, I, True, "softmax_normal")
    W = inputs.layer_weights(cfg, "cpu", fp4=True)
    g = torch.Generator().manual_seed(11)
    def spread(sc):
        delta = torch.randint(-20, 21, sc.shape, generator=g, dtype=torch.int32)
        return (sc.to(torch.int32) + delta).clamp(1, 254).to(torch.uint8)
    for n in ("s_gate", "s_up", "s_down"):
        W[n] = spread(W[n])
    sh = list(W["shared"])
    for i in (1, 3, 5):
        sh[i] = spread(sh[i])
    W["shared"] = tuple(sh)
    Wd = _dev_weights(W, cuda_device)
    x, ids, w = inputs.layer_batch(cfg, 5)
    _compare(cuda_device, W, Wd, x, ids, w, range(5), f"fp4 wide scales {E},{k},{d},{I}")


@pytest.mark.parametrize("E,k,d,I", [(4, 2, 512, 256), (3, 3, 1056, 64)])
def test_fp4_scale_exponents_at_the_ends(cuda_device, E, k, d, I):
    """Some blocks' scale bytes at the bottom of the E8M0 range (1..4: the
    scaled partial sums are FP32 subnormals or nearly) and some 21..26 above
    the rest (the block dominates its dot product; larger steps would take y
    past the FP32 range), on both kernel families:
    each block's scale multiplies its own partial sum, and the routing weight
    the expert's whole dot, as the oracle computes them."""
    cfg = inputs.LayerConfig(f"fp4_ends_{E}_{k}_{d}_{I}", E, k, d, I, True, "softmax_normal")
    W = inputs.layer_weights(cfg, "cpu", fp4=True)
    g = torch.Generator().manual_seed(12)
    def ends(sc):
        u = torch.rand(sc.shape, generator=g)
        low = torch.randint(1, 5, sc.shape, generator=g, dtype=torch.int32)
        high = sc.to(torch.int32) + torch.randint(21, 27, sc.shape, generator=g, dtype=torch.int32)
        out = torch.where(u < 0.1, low, torch.where(u > 0.95, high.clamp(max=254), sc.to(torch.int32)))
        return out.to(torch.uint8)
    for n in ("s_gate", "s_up", "s_down"):
        W[n] = ends(W[n])
    sh = list(W["shared"])
    for i in (1, 3, 5):
        sh[i] = ends(sh[i])
    W["shared"] = tuple(sh)
    Wd = _dev_weights(W, cuda_device)
    x, ids, w = inputs.layer_batch(cfg, 5)
    _compare(cuda_device, W, Wd, x, ids, w, range(5), f"fp4 end scales {E},{k},{d},{I}")


@pytest.mark.parametrize("E,k,d,I", [(5, 2, 96, 160), (3, 3, 1056, 64)])
def test_fp4_shared_expert_and_ragged_lanes(cuda_device, E, k, d, I):
    """A shared expert; rows whose chunk count is not a multiple of 32."""
    cfg = inputs.LayerConfig(f"fp4_edge_{E}_{k}_{d}_{I}", E, k, d, I, True, "softmax_normal")
    W = inputs.layer_weights(cfg, "cpu", fp4=True)
    Wd = _dev_weights(W, cuda_device)
    x, ids, w = inputs.layer_batch(cfg, 5)
    _compare(cuda_device, W, Wd, x, ids, w, range(5), f"fp4 edge {E},{k},{d},{I}")


def test_fp4_bad_expert_id_sets_flag_and_skips_slot(cuda_device):
    W = inputs.layer_weights(inputs.TINY, "cpu", fp4=True)
    Wd = _dev_weights(W, cuda_device)
    x, ids, w = inputs.layer_batch(inputs.TINY, 4)
    bad = ids.clone()
    bad[2, 1] = inputs.TINY.E
    moe.device_error(cuda_device)
    _, y = _run(cuda_device, Wd, x, bad, w)
    assert moe.device_error(cuda_device) & 1
    fixed, w0 = ids.clone(), w.clone()
    fixed[2, 1] = 0
    w0[2, 1] = 0.0
    ref = _oracle(W, x, fixed, w0, range(4))
    check_close(y, ref["y64"], "fp4 bad id")
    assert moe.device_error(cuda_device) == 0
