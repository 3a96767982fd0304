"""CPU oracle for the MoE decode layer and moe_align_block_size.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's cpu_baseline / reference legs, never by the library.  It shares
no code with the CUDA path; the C source (moe_oracle.c) is the oracle, this
module only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_decode.restype = ctypes.c_double
        lib.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_moe_layer.restype = ctypes.c_int
        lib.oracle_moe_layer.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
                                         P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                         P, P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_moe_layer_mx4.restype = ctypes.c_int
        lib.oracle_moe_layer_mx4.argtypes = lib.oracle_moe_layer.argtypes
        lib.oracle_e2m1_decode.restype = ctypes.c_double
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_moe_layer_mx_act.restype = ctypes.c_int
        lib.oracle_moe_layer_mx_act.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
                                                P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_mx_requant.restype = ctypes.c_int
        lib.oracle_mx_requant.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P]
        lib.oracle_e4m3_round.restype = ctypes.c_double
        lib.oracle_e4m3_round.argtypes = [ctypes.c_double]
        lib.oracle_align_sizes.restype = ctypes.c_int
        lib.oracle_align_sizes.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int64)] * 2
        lib.oracle_router_topk.restype = ctypes.c_int
        lib.oracle_router_topk.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, P, P]
        lib.oracle_align.restype = ctypes.c_int
        lib.oracle_align.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     P, ctypes.c_int64, P, ctypes.c_int64, P]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def e4m3_decode(q: int) -> float:
    return _load().oracle_e4m3_decode(int(q))


def e8m0_decode(s: int) -> float:
    return _load().oracle_e8m0_decode(int(s))


def bf16_round(v: float) -> int:
    """BF16 bit pattern nearest to v (ties to even)."""
    return int(_load().oracle_bf16_round(float(v)))


def bf16_to_float(b: int) -> float:
    return _load().oracle_bf16_to_double(int(b))


def e2m1_decode(q: int) -> float:
    """Value of one FP4 E2M1 code (low 4 bits of q)."""
    return float(_load().oracle_e2m1_decode(q & 15))


def moe_layer(x_bf16, topk_ids, topk_w, w_gate, s_gate, w_up, s_up, w_down, s_down,
              shared=None, want_truth=False, fp4=False):
    """Run the FP64 oracle layer.

    x_bf16: uint16 [B, d] (BF16 bit patterns); topk_ids int32 [B, k];
    topk_w float32 [B, k]; w_* uint8 [E, rows, K] E4M3 codes; s_* uint8
    [E, rows, K/32] E8M0 scales; shared: None or a 6-tuple
    (w_gate, s_gate, w_up, s_up, w_down, s_down) with a leading dim of 1.
    Returns dict(h=uint16 [B, k+S, I] (BF16 bits), h64=float64 [B, k+S, I]
    (unrounded intermediates), g64/u64 (the gate and up dots), y64=float64
    [B, d], truth64=... ).  fp4=True: MXFP4 weights, w_* uint8 [E, rows,
    K/2] with two E2M1 codes per byte (the lower K index in the low nibble).
    """
    lib = _load()
    x = _c(x_bf16, np.uint16)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    B, d = x.shape
    k = ids.shape[1] if ids.ndim == 2 else 0
    wg, sg, wu, su = (_c(a, np.uint8) for a in (w_gate, s_gate, w_up, s_up))
    wd, sd = _c(w_down, np.uint8), _c(s_down, np.uint8)
    E, I = wg.shape[0], wg.shape[1]
    cw = 2 if fp4 else 1
    assert wg.shape == (E, I, d // cw) and wu.shape == (E, I, d // cw) and wd.shape == (E, d, I // cw)
    assert sg.shape == (E, I, d // 32) and su.shape == (E, I, d // 32) and sd.shape == (E, d, I // 32)
    sh = [None] * 6
    S = 0
    if shared is not None:
        sh = [_c(a, np.uint8) for a in shared]
        S = 1
    h = np.zeros((B, k + S, I), dtype=np.uint16)
    h64 = np.zeros((B, k + S, I), dtype=np.float64)
    g64 = np.zeros((B, k + S, I), dtype=np.float64)
    u64 = np.zeros((B, k + S, I), dtype=np.float64)
    y = np.zeros((B, d), dtype=np.float64)
    t = np.zeros((B, d), dtype=np.float64) if want_truth else None
    fn = lib.oracle_moe_layer_mx4 if fp4 else lib.oracle_moe_layer
    rc = fn(_ptr(x), B, d, _ptr(ids), _ptr(w), k, _ptr(wg), _ptr(sg), _ptr(wu),
            _ptr(su), _ptr(wd), _ptr(sd), E, I, *(_ptr(a) for a in sh),
            _ptr(h), _ptr(h64), _ptr(g64), _ptr(u64), _ptr(y), _ptr(t))
    if rc != 0:
        raise ValueError(f"oracle_moe_layer rejected its arguments (rc={rc})")
    out = {"h": h, "h64": h64, "g64": g64, "u64": u64, "y64": y}
    if want_truth:
        out["truth64"] = t
    return out


def moe_layer_mx_act(x_bf16, topk_ids, topk_w, w_gate, s_gate, w_up, s_up, w_down, s_down,
                     shared=None):
    """The conventional path's numerics: moe_layer with x and h converted to
    MXFP8 and back before their GEMMs (see mx_requant).  Same arguments as
    moe_layer; returns dict(h, h64, g64, u64, y64) of the converted-x pass."""
    lib = _load()
    x = _c(x_bf16, np.uint16)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    B, d = x.shape
    k = ids.shape[1] if ids.ndim == 2 else 0
    wg, sg, wu, su = (_c(a, np.uint8) for a in (w_gate, s_gate, w_up, s_up))
    wd, sd = _c(w_down, np.uint8), _c(s_down, np.uint8)
    E, I = wg.shape[0], wg.shape[1]
    assert wg.shape == (E, I, d) and wu.shape == (E, I, d) and wd.shape == (E, d, I)
    sh = [None] * 6
    S = 0
    if shared is not None:
        sh = [_c(a, np.uint8) for a in shared]
        S = 1
    h = np.zeros((B, k + S, I), dtype=np.uint16)
    h64 = np.zeros((B, k + S, I), dtype=np.float64)
    g64 = np.zeros((B, k + S, I), dtype=np.float64)
    u64 = np.zeros((B, k + S, I), dtype=np.float64)
    y = np.zeros((B, d), dtype=np.float64)
    rc = lib.oracle_moe_layer_mx_act(_ptr(x), B, d, _ptr(ids), _ptr(w), k, _ptr(wg), _ptr(sg), _ptr(wu),
                                     _ptr(su), _ptr(wd), _ptr(sd), E, I, *(_ptr(a) for a in sh),
                                     _ptr(h), _ptr(h64), _ptr(g64), _ptr(u64), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_moe_layer_mx_act rejected its arguments (rc={rc})")
    return {"h": h, "h64": h64, "g64": g64, "u64": u64, "y64": y}


def e4m3_round(q: float) -> float:
    """The E4M3 value nearest q (ties to the even code, saturating at 448)."""
    return float(_load().oracle_e4m3_round(float(q)))


def mx_requant(x_bf16) -> np.ndarray:
    """BF16 -> MXFP8 (OCP MX v1.0: shared exponent floor(log2 max|v|) - 8 per
    32 values along the last axis, E4M3 elements nearest-even, saturating)
    -> BF16.  x_bf16: uint16 [..., K] BF16 bit patterns, K % 32 == 0."""
    x = _c(x_bf16, np.uint16)
    K = x.shape[-1]
    rows = x.size // K if K else 0
    out = np.zeros_like(x)
    rc = _load().oracle_mx_requant(_ptr(x), rows, K, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_mx_requant rejected its arguments (rc={rc})")
    return out


def align_sizes(T: int, k: int, E: int, block_size: int):
    n_sorted, n_blocks = ctypes.c_int64(), ctypes.c_int64()
    rc = _load().oracle_align_sizes(T, k, E, block_size, ctypes.byref(n_sorted), ctypes.byref(n_blocks))
    if rc != 0:
        raise ValueError("bad align sizes")
    return n_sorted.value, n_blocks.value


def align(topk_ids, E: int, block_size: int):
    """Stable counting sort by expert with block padding (see moe_oracle.c)."""
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    n_sorted, n_blocks = align_sizes(T, k, E, block_size)
    sorted_ids = np.empty(n_sorted, dtype=np.int32)
    expert_ids = np.empty(n_blocks, dtype=np.int32)
    ntpp = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_align(_ptr(ids), T, k, E, block_size, _ptr(sorted_ids), n_sorted,
                              _ptr(expert_ids), n_blocks, _ptr(ntpp))
    if rc != 0:
        raise ValueError(f"oracle_align rejected its arguments (rc={rc})")
    return sorted_ids, expert_ids, int(ntpp[0])


def router_topk(logits, k: int, score: str = "softmax", scale: float = 1.0):
    """Routing by definition (see moe_oracle.c): logits float32 [B, E] ->
    (ids int32 [B, k], w float64 [B, k]); score "softmax" or "sigmoid"."""
    lg = _c(logits, np.float32)
    B, E = lg.shape
    ids = np.empty((B, k), dtype=np.int32)
    w = np.empty((B, k), dtype=np.float64)
    rc = _load().oracle_router_topk(_ptr(lg), B, E, k, {"softmax": 0, "sigmoid": 1}[score], float(scale),
                                    _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle_router_topk rejected its arguments (rc={rc})")
    return ids, w
