"""GPU moe_align_block_size against the CPU oracle: bit-exact, every output."""
import json
import os

import numpy as np
import pytest
import torch

import mixture_experts_decode_gb300 as moe
import oracle
from mixture_experts_decode_gb300 import inputs

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gpu_align(ids_cpu, E, bs, dev):
    s, e, n = moe.align_block_size(ids_cpu.to(dev), E, bs)
    torch.cuda.synchronize()
    return s.cpu().numpy(), e.cpu().numpy(), int(n.item())


def _assert_exact(ids_cpu, E, bs, dev):
    s, e, n = _gpu_align(ids_cpu, E, bs, dev)
    rs, re_, rn = oracle.align(ids_cpu.numpy(), E, bs)
    assert n == rn
    assert np.array_equal(e, re_), "expert_ids differ"
    if not np.array_equal(s, rs):
        bad = np.nonzero(s != rs)[0]
        raise AssertionError(f"sorted_token_ids differ at {bad.size} positions, first {bad[:8]}")
    assert moe.device_error(dev) == 0


@pytest.mark.parametrize("routing", ["softmax_normal", "zipf"])
def test_prefill_scale_bit_exact(cuda_device, routing):
    # T=16384 tokens x top-8 of E=256, block_size 64
    ids = inputs.align_ids(16384, 8, 256, routing)
    _assert_exact(ids, 256, 64, cuda_device)


def test_golden_cases(cuda_device):
    with open(os.path.join(GOLDEN, "align_tiny.json")) as f:
        for c in json.load(f)["cases"]:
            s, e, n = _gpu_align(torch.tensor(c["topk_ids"], dtype=torch.int32), c["E"],
                                 c["block_size"], cuda_device)
            assert s.tolist() == c["sorted_token_ids"]
            assert e.tolist() == c["expert_ids"]
            assert n == c["num_tokens_post_pad"]


@pytest.mark.parametrize("T,k,E,bs", [(1, 1, 1, 1), (5, 3, 7, 2), (33, 8, 16, 16), (9, 8, 8, 4096),
                                      (1000, 6, 64, 1), (4099, 2, 1024, 64), (100000, 8, 256, 64),
                                      (777, 8, 513, 128)])
def test_shapes_bit_exact(cuda_device, T, k, E, bs):
    ids = inputs.align_ids(T, k, E, "softmax_normal", step=T + E)
    _assert_exact(ids, E, bs, cuda_device)


def test_one_hot_expert_and_empty(cuda_device):
    _assert_exact(torch.full((3000, 4), 5, dtype=torch.int32), 8, 64, cuda_device)
    _assert_exact(torch.empty((0, 4), dtype=torch.int32), 8, 16, cuda_device)


def test_bad_id_sets_flag_and_is_dropped(cuda_device):
    ids = inputs.align_ids(257, 4, 16, "softmax_normal")
    bad = ids.clone()
    bad[100, 2] = 16
    moe.device_error(cuda_device)
    s, e, n = _gpu_align(bad, 16, 8, cuda_device)
    assert moe.device_error(cuda_device) & 1
    N = 257 * 4
    # expected: the stable sort of every valid flat index, the bad one absent
    flat = bad.reshape(-1).numpy()
    valid = [f for f in range(N) if 0 <= flat[f] < 16]
    got = s[s < N]
    assert sorted(got.tolist()) == valid
    cnt = np.bincount(flat[valid], minlength=16)
    assert n == int(np.sum((cnt + 7) // 8 * 8))


def test_graph_capture(cuda_device):
    dev = cuda_device
    T, k, E, bs = 4096, 8, 128, 32
    ids = inputs.align_ids(T, k, E).to(dev)
    ns, nb, wsb = moe.align_sizes(T, k, E, bs)
    s = torch.empty(ns, dtype=torch.int32, device=dev)
    e = torch.empty(nb, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    moe.align_block_size(ids, E, bs, s, e, n, ws)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.align_block_size(ids, E, bs, s, e, n, ws)
    new = inputs.align_ids(T, k, E, "zipf")
    ids.copy_(new.to(dev))
    g.replay()
    torch.cuda.synchronize()
    rs, re_, rn = oracle.align(new.numpy(), E, bs)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(e.cpu().numpy(), re_)
    assert int(n.item()) == rn


@pytest.mark.parametrize("nbytes", [32, 32 * 257, 1 << 22])
def test_copy_kernel(cuda_device, nbytes):
    """One 32-byte element, a ragged last CTA (257 elements), 4 MiB; the
    bytes after the copied span stay untouched."""
    gen = torch.Generator(device=cuda_device).manual_seed(nbytes)
    src = torch.randint(0, 255, (nbytes + 4096,), dtype=torch.uint8, device=cuda_device, generator=gen)
    dst = torch.full_like(src, 0xA5)
    moe.copy(dst[:nbytes], src[:nbytes])
    torch.cuda.synchronize()
    assert torch.equal(dst[:nbytes], src[:nbytes])
    assert bool((dst[nbytes:] == 0xA5).all())
