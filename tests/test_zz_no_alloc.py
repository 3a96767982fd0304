"""moe_align_block_size_static: the align entry point for callers that cannot
hand the library any device scratch memory (engines that forbid allocation
after start-up, plugin hosts that pass only inputs and outputs, code that may
run during stream capture).  Its scratch is a fixed array inside the
library, so the test checks, through the C ABI, that two calls in a row give
exactly what the workspace-taking moe_align_block_size gives.

This file is collected last on purpose: it must pass on its own in a fresh
process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_decode_gb300 as moe
from mixture_experts_decode_gb300 import _lib, inputs


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(lib, ids, E, bs, dev):
    T, k = ids.shape
    ns, nb, _ = moe.align_sizes(T, k, E, bs)
    # poison the outputs so a missed write shows up
    s = torch.full((ns,), -7, dtype=torch.int32, device=dev)
    e = torch.full((nb,), -7, dtype=torch.int32, device=dev)
    n = torch.full((1,), -7, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = lib.moe_align_block_size_static(_ptr(ids), T, k, E, bs, _ptr(s), _ptr(e), _ptr(n), stream)
    assert rc == 0, lib.moe_strerror(rc).decode()
    return s, e, n


def _workspace_call(lib, ids, E, bs, dev):
    T, k = ids.shape
    ns, nb, wsb = moe.align_sizes(T, k, E, bs)
    s = torch.empty(ns, dtype=torch.int32, device=dev)
    e = torch.empty(nb, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = lib.moe_align_block_size(_ptr(ids), T, k, E, bs, _ptr(s), _ptr(e), _ptr(n), _ptr(ws),
                                  ws.numel(), stream)
    assert rc == 0, lib.moe_strerror(rc).decode()
    return s, e, n


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice():
    assert torch.cuda.is_available(), "needs a GPU"
    dev = torch.device("cuda", 0)
    lib = moe.load()
    # the prefill-scale shape, then a different routing and shape, back to back
    cases = [(inputs.align_ids(16384, 8, 256, "softmax_normal"), 256, 64),
             (inputs.align_ids(3000, 6, 200, "zipf", step=1), 200, 16)]
    for ids_cpu, E, bs in cases:
        assert lib.moe_align_static_fits(ids_cpu.shape[0], ids_cpu.shape[1], E) == 1
        ids = ids_cpu.to(dev)
        got = _static_call(lib, ids, E, bs, dev)
        ref = _workspace_call(lib, ids, E, bs, dev)
        torch.cuda.synchronize()
        for g, r, name in zip(got, ref, ("sorted_token_ids", "expert_ids", "num_tokens_post_pad")):
            assert torch.equal(g, r), f"{name} differs from moe_align_block_size"
    assert moe.device_error(dev) == 0


def test_static_scratch_rejects_problems_beyond_its_size():
    lib = moe.load()
    # E=1024 with 160000 slots needs 79 chunks x 1024 experts x 4 B > 256 KB
    assert lib.moe_align_static_fits(20000, 8, 1024) == 0
    rc = lib.moe_align_block_size_static(ctypes.c_void_p(0x1000), 20000, 8, 1024, 64,
                                         ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000),
                                         ctypes.c_void_p(0x4000), None)
    assert rc == -3          # MOE_ERR_LIMIT, before touching the device
    assert "limit" in lib.moe_strerror(rc).decode()
    assert "moe_align_block_size_static" in _lib.EXPORTS
