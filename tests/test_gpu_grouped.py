"""GPU parity of the expert-centric layer (moe_layer_grouped: align, grouped
tensor-core GEMMs, combine) against the CPU oracle, through the C-ABI.

The tensor cores sum in their own order, so y is held to the plain bar of
the decode layer, |gpu - y64| <= 4e-3 * max(1, |y64|), and a per-token
cosine of 0.99999 against the oracle's unrounded FP64 y; act_mx=True
against the oracle variant that rounds x and h through MXFP8.  At
DeepSeek-V3 sizes (K = 7168, |y| up to ~20, where BF16 rounding of y alone
takes 3.9e-3 of the 4e-3) the bar holds beyond the bound of FP32 tensor-core
summation, derived from the oracle's values (tc_y_allowance)."""
import numpy as np
import pytest
import torch

import mixture_experts_decode_gb300 as moe
from mixture_experts_decode_gb300 import inputs

from _gpu_helpers import (_report, check_cosine, check_plain, device_mx, item_cover, oracle_tokens, small_weights,
                          tc_y_allowance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwen(cuda_device):
    W = inputs.layer_weights(inputs.QWEN3, cuda_device)
    return W, device_mx(W, cuda_device)


def run_grouped(dev, Wd, x, ids, w, act_mx=False):
    return moe.layer_grouped(x.to(dev), ids.to(dev), w.to(dev), Wd["gate"], Wd["up"], Wd["down"],
                             shared=Wd.get("shared"), act_mx=act_mx)


def compare_grouped(dev, W, Wd, x, ids, w, tokens, what, act_mx=False, chunk=8, tc_bound=False):
    """y against the oracle on `tokens`: the plain bar, or with tc_bound (long
    dot products, |y| > 1) the plain bar beyond the tensor-core summation
    allowance of tc_y_allowance; the per-token cosine always."""
    y = run_grouped(dev, Wd, x, ids, w, act_mx)
    torch.cuda.synchronize()
    assert moe.device_error(dev) == 0
    tokens = list(tokens)
    worst, cos_min, n_gap = 0.0, 1.0, 0
    d = y.shape[1]
    for c0 in range(0, len(tokens), chunk):
        toks = tokens[c0:c0 + chunk]
        ref = oracle_tokens(W, x, ids, w, toks, mx_act=act_mx)
        yt = y.index_select(0, torch.tensor(toks, dtype=torch.long, device=dev))
        allow = None
        if tc_bound:
            K_gu, K_dn = W["w_gate"].shape[2], W["w_down"].shape[2]
            allow, g = tc_y_allowance(W, ids[toks].cpu().numpy(), w[toks].cpu().numpy(), ref,
                                      x[toks].float().double().numpy(), d, K_gu, K_dn)
            n_gap += g
        worst = max(worst, check_plain(yt, ref["y64"], what + " y", allow))
        cos_min = min(cos_min, check_cosine(yt, ref["y64"], what + " y"))
    how = "asserted beyond the tensor-core summation allowance" if tc_bound else "asserted"
    _report(f"{what}: tokens {len(tokens)}/{x.shape[0]}, max plain scaled error {worst:.3e} ({how}), "
            f"min cosine {cos_min:.8f}" + (f", h with two valid roundings {n_gap}" if tc_bound else ""))
    return y


def expert_cover(ids):
    """Tokens such that every (expert, block of 128 of its slots in sorted
    order) holds at least one of them."""
    return item_cover(np.asarray(ids), False, tc=128)


@pytest.mark.parametrize("T", [1, 37, 700])
@pytest.mark.parametrize("act_mx", [False, True])
def test_grouped_small_every_token(cuda_device, T, act_mx):
    """E=8, d=256, I=256: at T=700 each expert has 175 slots on average --
    two blocks of 128 per expert, the second ragged."""
    W = small_weights(8, 256, 256, False, 11)
    Wd = device_mx(W, cuda_device)
    ids, w = inputs.route("softmax_normal", T, 8, 2, "grouped-small", T)
    x = inputs.randn((T, 256), "cpu", "grouped-small-x", T).to(torch.bfloat16)
    compare_grouped(cuda_device, W, Wd, x, ids, w, range(T), f"grouped small T={T} act_mx={act_mx}", act_mx)


@pytest.mark.parametrize("T", [37, 300])
@pytest.mark.parametrize("act_mx", [False, True])
def test_grouped_shared_expert_every_token(cuda_device, T, act_mx):
    """A shared expert: its pass covers every token in blocks of 128 (three
    at T = 300, the last ragged) and adds with weight 1 after the routed
    slots."""
    W = small_weights(8, 256, 256, True, 14)
    Wd = device_mx(W, cuda_device)
    ids, w = inputs.route("softmax_normal", T, 8, 2, "grouped-shared", T)
    x = inputs.randn((T, 256), "cpu", "grouped-shared-x", T).to(torch.bfloat16)
    compare_grouped(cuda_device, W, Wd, x, ids, w, range(T), f"grouped shared T={T} act_mx={act_mx}", act_mx)


def test_grouped_deepseek_sampled_tokens(cuda_device):
    """DeepSeek-V3 shapes (E=256 + shared, d=7168, I=2048) at B=64: the first
    16 tokens of a cover of every expert block (98 of the 225 distinct
    experts and the shared expert's first block); the host-side bound of the
    check costs seconds per token at these sizes."""
    W = inputs.layer_weights(inputs.DEEPSEEK_V3, cuda_device)
    Wd = device_mx(W, cuda_device)
    x, ids, w = inputs.layer_batch(inputs.DEEPSEEK_V3, 64)
    compare_grouped(cuda_device, W, Wd, x, ids, w, expert_cover(ids)[:16], "grouped deepseek B=64", chunk=4,
                    tc_bound=True)
    del W, Wd
    torch.cuda.empty_cache()


def test_grouped_hot_expert_many_blocks(cuda_device):
    """Every token picks expert 3: 600 slots of one expert = 5 blocks, the
    last ragged; the other slot spreads over the rest."""
    T = 600
    W = small_weights(8, 256, 256, False, 12)
    Wd = device_mx(W, cuda_device)
    ids, w = inputs.route("softmax_normal", T, 8, 2, "grouped-hot", T)
    ids[:, 0] = 3
    ids[:, 1] = torch.where(ids[:, 1] == 3, torch.full_like(ids[:, 1], 5), ids[:, 1])
    x = inputs.randn((T, 256), "cpu", "grouped-hot-x", T).to(torch.bfloat16)
    compare_grouped(cuda_device, W, Wd, x, ids, w, range(0, T, 3), "grouped hot expert T=600")


@pytest.mark.parametrize("B", [8, 32])
def test_grouped_qwen_every_token(cuda_device, qwen, B):
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    compare_grouped(cuda_device, W, Wd, x, ids, w, range(B), f"grouped qwen B={B}")


@pytest.mark.parametrize("B,routing", [(256, None), (1024, None), (256, "zipf")])
def test_grouped_qwen_expert_cover(cuda_device, qwen, B, routing):
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B, routing)
    toks = expert_cover(ids)
    compare_grouped(cuda_device, W, Wd, x, ids, w, toks, f"grouped qwen B={B} {routing or 'default'} routing")


def test_grouped_qwen_act_mx(cuda_device, qwen):
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, 64)
    compare_grouped(cuda_device, W, Wd, x, ids, w, expert_cover(ids), "grouped qwen B=64 act_mx", act_mx=True)


def test_grouped_bad_expert_id_sets_flag_and_skips_slot(cuda_device):
    W = small_weights(8, 256, 256, False, 13)
    Wd = device_mx(W, cuda_device)
    T = 40
    ids, w = inputs.route("softmax_normal", T, 8, 2, "grouped-bad", T)
    x = inputs.randn((T, 256), "cpu", "grouped-bad-x", T).to(torch.bfloat16)
    bad = ids.clone()
    bad[5, 1] = 8
    bad[17, 0] = -1
    moe.device_error(cuda_device)
    y = run_grouped(cuda_device, Wd, x, bad, w)
    assert moe.device_error(cuda_device) & 1
    fixed, w0 = ids.clone(), w.clone()
    fixed[5, 1], w0[5, 1] = 0, 0.0
    fixed[17, 0], w0[17, 0] = 0, 0.0
    ref = oracle_tokens(W, x, fixed, w0, range(T))
    check_plain(y, ref["y64"], "grouped bad id")
    assert moe.device_error(cuda_device) == 0


def test_grouped_empty_batch_is_noop(cuda_device, qwen):
    _, Wd = qwen
    x = torch.empty((0, 2048), dtype=torch.bfloat16, device=cuda_device)
    ids = torch.empty((0, 8), dtype=torch.int32, device=cuda_device)
    w = torch.empty((0, 8), dtype=torch.float32, device=cuda_device)
    y = moe.layer_grouped(x, ids, w, Wd["gate"], Wd["up"], Wd["down"])
    assert y.shape == (0, 2048)


def test_grouped_deterministic(cuda_device, qwen):
    _, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, 128)
    a = run_grouped(cuda_device, Wd, x, ids, w)
    b = run_grouped(cuda_device, Wd, x, ids, w)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
