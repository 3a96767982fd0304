"""C-ABI library on the host (no GPU needed): it loads, exports every symbol
include/moedec.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import mixture_experts_decode_gb300 as moe
from mixture_experts_decode_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moedec.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_decode_gb300 import build
    build.build()
    return moe.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    assert lib.moe_version() >= 100
    for code in range(0, -8, -1):
        assert lib.moe_strerror(code).decode()
    assert lib.moe_strerror(-99).decode() == "unknown status"


def _mx(addr=0x10000):
    return _lib.MXView(addr, addr)


def _gate_up(lib, B=2, d=64, k=2, E=4, I=64, x=0x20000, ids=0x30000, h=0x40000, w=0x10000):
    return lib.moe_gate_up(x, B, d, ids, k, _mx(w), _mx(w), E, I, None, None, h, None)


def test_gate_up_rejects_bad_shapes_before_launch(lib):
    assert _gate_up(lib, d=33) == -2
    assert _gate_up(lib, I=48) == -2
    assert _gate_up(lib, k=5, E=4) == -2
    assert _gate_up(lib, B=-1) == -1
    assert _gate_up(lib, B=257) == -3
    assert _gate_up(lib, B=256, k=9, E=16) == -3
    assert _gate_up(lib, E=1025, k=2) == -3
    assert _gate_up(lib, x=0) == -1
    assert _gate_up(lib, x=0x20010) == -5                # not 32-byte aligned
    assert _gate_up(lib, w=0x10010) == -5
    assert _gate_up(lib, B=0, x=0) == 0                  # empty batch: no-op, no launch


def test_down_and_layer_reject_bad_arguments(lib):
    m = _mx()
    assert lib.moe_down(0x40000, 2, 2, 0x30000, 0x50000, m, 4, 64, 40, None, 0x60000, None) == -2
    assert lib.moe_down(0x40000, 2, 2, 0x30000, None, m, 4, 64, 64, None, 0x60000, None) == -1
    ws = ctypes.c_size_t()
    assert lib.moe_layer_workspace_bytes(4, 8, 768, 1, ctypes.byref(ws)) == 0
    assert ws.value == 4 * 9 * 768 * 4                  # FP32 intermediate, [B][k+S][I]
    assert lib.moe_layer_workspace_bytes(4, 8, 768, 0, ctypes.byref(ws)) == 0
    small = ws.value - 1
    rc = lib.moe_layer(0x20000, 4, 2048, 0x30000, 0x50000, 8, m, m, m, 16, 768, None, None, None,
                       0x70000, small, 0x60000, None)
    assert rc == -4
    sh = ctypes.byref(m)
    rc = lib.moe_layer(0x20000, 4, 2048, 0x30000, 0x50000, 8, m, m, m, 16, 768, sh, None, None,
                       0x70000, 1 << 30, 0x60000, None)
    assert rc == -1                                      # shared expert: all three or none


def test_align_sizes_and_checks(lib):
    ns, nb, wsb = moe.align_sizes(16384, 8, 256, 64)
    assert (ns, nb) == (147200, 2300)                   # T*k + E*(bs-1), ceil(/bs)
    assert wsb > 0
    assert lib.moe_align_sizes(4, 2, 1025, 8, None, None, None) == -3
    assert lib.moe_align_sizes(4, 2, 8, 0, None, None, None) == -1
    assert lib.moe_align_sizes(1 << 28, 8, 8, 8, None, None, None) == -3   # exceeds int32
    rc = lib.moe_align_block_size(0x30000, 16, 2, 8, 4, 0x40000, 0x50000, 0x60000, 0x70000, 0, None)
    assert rc == -4


def test_host_and_device_workspace_sizes(lib):
    assert moe.layer_host_workspace_bytes(32, 2048, 8, 768, False) >= \
        moe.layer_workspace_bytes(32, 8, 768, False) + 2 * 32 * 2048 * 2


def test_router_rejects_bad_arguments_before_launch(lib):
    P = ctypes.c_void_p
    good = (P(0x10000), P(0x20000), P(0x30000))
    assert lib.moe_router_topk(good[0], 4, 8, 9, 0, 1.0, good[1], good[2], None) == -2     # k > E
    assert lib.moe_router_topk(good[0], 4, 2048, 8, 0, 1.0, good[1], good[2], None) == -3  # E > max
    assert lib.moe_router_topk(good[0], 4, 64, 33, 0, 1.0, good[1], good[2], None) == -3   # k > max
    assert lib.moe_router_topk(good[0], 4, 64, 8, 2, 1.0, good[1], good[2], None) == -1    # score
    assert lib.moe_router_topk(good[0], -1, 64, 8, 0, 1.0, good[1], good[2], None) == -1   # B < 0
    assert lib.moe_router_topk(None, 4, 64, 8, 0, 1.0, good[1], good[2], None) == -1       # NULL
    assert lib.moe_router_topk(P(0x10002), 4, 64, 8, 0, 1.0, good[1], good[2], None) == -5  # alignment
    assert lib.moe_router_topk(None, 0, 64, 8, 1, 2.5, None, None, None) == 0               # B = 0


def test_mx_requant_rejects_bad_arguments_before_launch(lib):
    P = ctypes.c_void_p
    a, b = P(0x10000), P(0x20000)
    assert lib.moe_mx_requant(a, b, -1, 64, None) == -1           # rows < 0
    assert lib.moe_mx_requant(a, b, 4, 48, None) == -2            # K not a multiple of 32
    assert lib.moe_mx_requant(a, b, 4, 0, None) == -2             # K = 0
    assert lib.moe_mx_requant(a, b, 1 << 62, 1 << 20, None) == -3  # rows * K overflows
    assert lib.moe_mx_requant(None, b, 4, 64, None) == -1         # NULL
    assert lib.moe_mx_requant(a, P(0x20008), 4, 64, None) == -5   # 16-byte alignment
    assert lib.moe_mx_requant(None, None, 0, 64, None) == 0       # rows = 0 launches nothing


def test_fp4_passes_reject_bad_arguments_before_launch(lib):
    from mixture_experts_decode_gb300._lib import MXView
    P = ctypes.c_void_p
    mx = MXView(0x100000, 0x200000)
    x, ids, h, w, y = P(0x300000), P(0x400000), P(0x500000), P(0x600000), P(0x700000)
    assert lib.moe_gate_up_fp4(x, 4, 48, ids, 2, mx, mx, 8, 64, None, None, h, None) == -2      # d % 32
    assert lib.moe_gate_up_fp4(x, 4, 64, ids, 9, mx, mx, 8, 64, None, None, h, None) == -2      # k > E
    assert lib.moe_gate_up_fp4(x, 4, 64, ids, 2, mx, mx, 8, 64, ctypes.byref(mx), None, h, None) == -1
    assert lib.moe_gate_up_fp4(P(0x300008), 4, 64, ids, 2, mx, mx, 8, 64, None, None, h, None) == -5
    assert lib.moe_gate_up_fp4(None, 0, 64, None, 2, mx, mx, 8, 64, None, None, None, None) == 0  # B = 0
    assert lib.moe_down_fp4(h, 4, 2, ids, w, mx, 8, 64, 48, None, y, None) == -2                 # I % 32
    assert lib.moe_down_fp4(h, 4, 2, ids, None, mx, 8, 64, 64, None, y, None) == -1             # NULL
    assert lib.moe_down_fp4(P(0x500008), 4, 2, ids, w, mx, 8, 64, 64, None, y, None) == -5


def test_grouped_layer_rejects_bad_arguments_before_launch(lib):
    m = _mx()
    ws = ctypes.c_size_t()
    assert lib.moe_layer_grouped_workspace_bytes(256, 8, 128, 2048, 768, 0, ctypes.byref(ws)) == 0
    plain = ws.value
    ns = 256 * 8 + 128 * 127
    # at least the sort output, h for every sorted row and the FP32 per-slot outputs
    assert ws.value >= ns * 4 + ns * 768 * 2 + 256 * 8 * 2048 * 4
    assert lib.moe_layer_grouped_workspace_bytes(4, 2, 8, 96, 256, 0, ctypes.byref(ws)) == -2   # d % 128
    assert lib.moe_layer_grouped_workspace_bytes(4, 2, 8, 256, 160, 0, ctypes.byref(ws)) == -2  # I % 128
    assert lib.moe_layer_grouped_workspace_bytes(4, 9, 8, 256, 256, 0, ctypes.byref(ws)) == -2   # k > E
    assert lib.moe_layer_grouped_workspace_bytes(4, 2, 1025, 256, 256, 0, ctypes.byref(ws)) == -3
    assert lib.moe_layer_grouped_workspace_bytes(-1, 2, 8, 256, 256, 0, ctypes.byref(ws)) == -1

    assert lib.moe_layer_grouped_workspace_bytes(256, 8, 128, 2048, 768, 1, ctypes.byref(ws)) == 0
    # a shared expert adds its own sort, h rows (T rounded to 128) and FP32 rows
    assert ws.value >= plain + 256 * 768 * 2 + 256 * 2048 * 4

    def call(T=4, x=0x20000, ids=0x30000, w=0x40000, act=0, wsp=0x70000, wsb=1 << 40, y=0x60000,
             sg=None, su=None, sd=None):
        return lib.moe_layer_grouped(x, T, 256, ids, w, 2, m, m, m, 8, 256, sg, su, sd, act, wsp, wsb, y, None)

    assert call(act=2) == -1
    assert call(x=0) == -1
    assert call(x=0x20010) == -5                          # x not 32-byte aligned
    assert call(wsb=16) == -4
    assert call(wsp=0x70010) == -5                        # workspace not 256-byte aligned
    assert call(T=0, x=0) == 0                            # empty batch: no launch
    assert call(sg=ctypes.byref(m)) == -1                 # shared expert: all three or none
