"""GPU parity of the decode layer (moe_gate_up / moe_down / moe_layer) against
the CPU oracle, through the C-ABI.  Tolerance: see tests/_gpu_helpers.py."""
import numpy as np
import pytest
import torch

import mixture_experts_decode_gb300 as moe
from mixture_experts_decode_gb300 import inputs

from _gpu_helpers import (check_close, compare_tokens, device_mx, item_cover, oracle_tokens, run_gate_up,
                          run_layer, small_weights)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwen(cuda_device):
    W = inputs.layer_weights(inputs.QWEN3, cuda_device)
    return W, device_mx(W, cuda_device)


@pytest.fixture(scope="module")
def tiny(cuda_device):
    W = inputs.layer_weights(inputs.TINY, "cpu")
    return W, device_mx(W, cuda_device)


@pytest.mark.parametrize("B", [1, 3, 16])
def test_tiny_layer_full(cuda_device, tiny, B):
    W, Wd = tiny
    x, ids, w = inputs.layer_batch(inputs.TINY, B)
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"tiny B={B}")


@pytest.mark.parametrize("B", [1, 2, 4])
def test_qwen_full_batch(cuda_device, qwen, B):
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"qwen B={B}")


@pytest.mark.parametrize("B", [8, 16, 32])
def test_qwen_every_token(cuda_device, qwen, B):
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"qwen B={B}")


@pytest.mark.parametrize("routing", ["contiguous", "zipf", "softmax_uniform"])
def test_qwen_locality_routings(cuda_device, qwen, routing):
    """Every token of the B=32 batch under each routing of the locality sweep."""
    W, Wd = qwen
    B = 32
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B, routing=routing)
    if routing == "contiguous":
        assert inputs.unique_experts(ids) == 128
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"qwen B=32 {routing}")


@pytest.mark.parametrize("B", [64, 256])
def test_qwen_large_batch_item_cover(cuda_device, qwen, B):
    """Above the decode batches: one token of every (expert, 4-token group)
    work item, so every item of both passes meets the oracle."""
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    toks = item_cover(ids.numpy(), False)
    compare_tokens(cuda_device, W, Wd, x, ids, w, toks, f"qwen B={B} item cover")


@pytest.mark.parametrize("B,routing", [(32, None), (32, "zipf"), (64, None)])
def test_qwen_gate_up_every_tile(cuda_device, qwen, B, routing):
    """h of every token and slot: with experts that need more than one pass
    the gate/up tiles are dealt heaviest expert first, and each (expert, row
    block) must still be computed exactly once."""
    W, Wd = qwen
    kw = {} if routing is None else {"routing": routing}
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B, **kw)
    counts = torch.bincount(ids.reshape(-1).long(), minlength=inputs.QWEN3.E)
    assert int(counts.max()) > 4, "the batch must hold an expert with more than one pass"
    h = run_gate_up(cuda_device, Wd, x, ids)
    torch.cuda.synchronize()
    ref = oracle_tokens(W, x, ids, w, range(B))
    check_close(h, ref["h64"], f"qwen B={B} {routing} h")
    assert moe.device_error(cuda_device) == 0


@pytest.fixture(scope="module")
def deepseek(cuda_device):
    W = inputs.layer_weights(inputs.DEEPSEEK_V3, cuda_device)
    yield W, device_mx(W, cuda_device)
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [1, 8])
def test_deepseek_every_token(cuda_device, deepseek, B):
    W, Wd = deepseek
    x, ids, w = inputs.layer_batch(inputs.DEEPSEEK_V3, B)
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"deepseek B={B}", plain=False)


@pytest.mark.parametrize("B", [32, 64])
def test_deepseek_item_cover(cuda_device, deepseek, B):
    """One token of every (expert, 4-token group) item, the shared expert's
    groups included."""
    W, Wd = deepseek
    x, ids, w = inputs.layer_batch(inputs.DEEPSEEK_V3, B)
    toks = item_cover(ids.numpy(), True)
    compare_tokens(cuda_device, W, Wd, x, ids, w, toks, f"deepseek B={B} item cover", plain=False)


# (E, k, d, I, shared): lanes-per-row L = 1, 2, 4, 8, 16, 32 on both passes,
# rows that do not fill the last CTA, k = 1, k = E
EDGE_SHAPES = [(4, 1, 32, 32, False), (5, 2, 96, 160, False), (3, 3, 160, 64, True),
               (6, 2, 512, 96, True), (2, 2, 1024, 512, False), (7, 4, 64, 1056, True)]


@pytest.mark.parametrize("E,k,d,I,shared", EDGE_SHAPES)
def test_edge_shapes(cuda_device, E, k, d, I, shared):
    W = small_weights(E, d, I, shared, 1)
    Wd = device_mx(W, cuda_device)
    for B in (1, 5):
        cfg = inputs.LayerConfig("edge", E, k, d, I, shared, "softmax_normal")
        x, ids, w = inputs.layer_batch(cfg, B, step=E * 100 + d)
        compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"edge {E},{k},{d},{I},{shared} B={B}")


def _layer_with_canaries(dev, Wd, x, ids, w, shared):
    """Run moe_layer with y and the workspace cut out of larger buffers whose
    guard bytes hold a fixed pattern; returns y and whether every guard byte
    is still intact."""
    B, d = x.shape
    k = ids.shape[1]
    I = Wd["gate"].w.shape[1]
    G = 512  # guard bytes on each side (keeps both regions 512-byte aligned)
    need = moe.layer_workspace_bytes(B, k, I, shared)
    ws_buf = torch.full((need + 2 * G,), 0xA5, dtype=torch.uint8, device=dev)
    y_buf = torch.full((2 * B * d + 2 * G,), 0x5A, dtype=torch.uint8, device=dev)
    y = y_buf[G:G + 2 * B * d].view(torch.bfloat16).view(B, d)
    moe.layer(x.to(dev), ids.to(dev), w.to(dev), Wd["gate"], Wd["up"], Wd["down"], shared=Wd["shared"],
              workspace=ws_buf[G:G + need], y=y)
    torch.cuda.synchronize()
    intact = bool((ws_buf[:G] == 0xA5).all() and (ws_buf[G + need:] == 0xA5).all()
                  and (y_buf[:G] == 0x5A).all() and (y_buf[G + 2 * B * d:] == 0x5A).all())
    return y, intact


@pytest.mark.parametrize("B", [1, 3])
def test_outputs_stay_in_bounds_qwen(cuda_device, qwen, B):
    """The layer writes y [B][d] and h at the head of the workspace and no
    byte around them (the down pass's row blocks need not divide d)."""
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    y, intact = _layer_with_canaries(cuda_device, Wd, x, ids, w, False)
    assert intact, "a kernel wrote outside y or the workspace"
    assert torch.isfinite(y.float()).all()
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"qwen canary B={B}")


@pytest.mark.parametrize("E,k,d,I,shared", [(2, 2, 1024, 512, False), (5, 2, 1536, 768, True)])
def test_outputs_stay_in_bounds_edge(cuda_device, E, k, d, I, shared):
    W = small_weights(E, d, I, shared, 3)
    Wd = device_mx(W, cuda_device)
    for B in (1, 4):
        cfg = inputs.LayerConfig("canary", E, k, d, I, shared, "softmax_normal")
        x, ids, w = inputs.layer_batch(cfg, B, step=E * 10 + d)
        y, intact = _layer_with_canaries(cuda_device, Wd, x, ids, w, shared)
        assert intact, f"a kernel wrote outside y or the workspace ({E},{k},{d},{I},{shared}) B={B}"
        compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), f"canary {E},{k},{d},{I},{shared} B={B}")


@pytest.mark.parametrize("d,I", [(128, 64), (256, 256)])
def test_hot_expert_and_duplicates(cuda_device, d, I):
    """Every token on one expert (more tokens than one pass serves) and the
    same expert twice inside one token's top-k (summed independently); at
    I = 256 the down pass is the row-tile kernel."""
    E = 4
    W = small_weights(E, d, I, True, 2)
    Wd = device_mx(W, cuda_device)
    B, k = 13, 3
    x, _, _ = inputs.layer_batch(inputs.LayerConfig("hot", E, k, d, I, True, "softmax_normal"), B)
    ids = torch.zeros((B, k), dtype=torch.int32)
    ids[:, 1] = 2
    ids[::2, 2] = 0                       # duplicate of slot 0 on even tokens
    ids[1::2, 2] = 3
    w = torch.rand((B, k), generator=torch.Generator().manual_seed(5))
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(B), "hot/dup")


def test_max_slots(cuda_device):
    """B * k at the documented maximum (2048 slots, B = 256)."""
    E, k, d, I = 16, 8, 64, 64
    W = small_weights(E, d, I, False, 3)
    Wd = device_mx(W, cuda_device)
    x, ids, w = inputs.layer_batch(inputs.LayerConfig("max", E, k, d, I, False, "softmax_normal"), 256)
    compare_tokens(cuda_device, W, Wd, x, ids, w, range(256), "max slots")


def test_empty_batch_is_noop(cuda_device, tiny):
    _, Wd = tiny
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=cuda_device)
    ids = torch.empty((0, 2), dtype=torch.int32, device=cuda_device)
    w = torch.empty((0, 2), dtype=torch.float32, device=cuda_device)
    y = moe.layer(x, ids, w, Wd["gate"], Wd["up"], Wd["down"])
    assert y.shape == (0, 256)


def test_bad_expert_id_sets_flag_and_skips_slot(cuda_device, tiny):
    W, Wd = tiny
    B = 4
    x, ids, w = inputs.layer_batch(inputs.TINY, B)
    bad = ids.clone()
    bad[2, 1] = 8                          # == E: out of range
    moe.device_error(cuda_device)          # clear
    y = run_layer(cuda_device, Wd, x, bad, w)
    assert moe.device_error(cuda_device) & 1
    # the bad slot contributes nothing: same as a valid id with weight 0
    fixed, w0 = ids.clone(), w.clone()
    fixed[2, 1] = 0
    w0[2, 1] = 0.0
    ref = oracle_tokens(W, x, fixed, w0, range(B))
    check_close(y, ref["y64"], "bad id")
    assert moe.device_error(cuda_device) == 0


@pytest.mark.parametrize("B", [8, 32])
def test_separate_passes_equal_layer(cuda_device, qwen, B):
    """moe_layer (FP32 intermediate in the down pass's order) and the two
    passes through the interface (BF16 h) give the same bits."""
    W, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, B)
    dev = cuda_device
    y1 = run_layer(dev, Wd, x, ids, w)
    h = run_gate_up(dev, Wd, x, ids)
    y2 = moe.down(h, ids.to(dev), w.to(dev), Wd["down"])
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_deterministic(cuda_device, qwen):
    _, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, 32)
    a = run_layer(cuda_device, Wd, x, ids, w)
    b = run_layer(cuda_device, Wd, x, ids, w)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_layer_host_matches_device_layer(cuda_device, qwen):
    _, Wd = qwen
    x, ids, w = inputs.layer_batch(inputs.QWEN3, 16)
    ref = run_layer(cuda_device, Wd, x, ids, w)
    xh, ih, wh = x.pin_memory(), ids.pin_memory(), w.pin_memory()
    y = moe.layer_host(xh, ih, wh, Wd["gate"], Wd["up"], Wd["down"])
    torch.cuda.synchronize()
    assert torch.equal(y, ref.cpu())


def test_cuda_graph_replay(cuda_device, qwen):
    _, Wd = qwen
    dev = cuda_device
    B = 32
    x0, i0, w0 = inputs.layer_batch(inputs.QWEN3, B, step=1)
    x, ids, w = x0.to(dev), i0.to(dev), w0.to(dev)
    ws = torch.empty(moe.layer_workspace_bytes(B, 8, 768, False), dtype=torch.uint8, device=dev)
    y = torch.empty((B, 2048), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        moe.layer(x, ids, w, Wd["gate"], Wd["up"], Wd["down"], workspace=ws, y=y)   # warm-up
    torch.cuda.current_stream(dev).wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.layer(x, ids, w, Wd["gate"], Wd["up"], Wd["down"], workspace=ws, y=y)
    for step in (2, 3):
        xs, is_, ws_ = inputs.layer_batch(inputs.QWEN3, B, step=step)
        x.copy_(xs.to(dev)); ids.copy_(is_.to(dev)); w.copy_(ws_.to(dev))
        g.replay()
        ref = run_layer(dev, Wd, xs, is_, ws_)
        torch.cuda.synchronize()
        assert torch.equal(y, ref)
