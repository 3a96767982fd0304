"""ctypes binding of libmoedec.so: argument marshalling only.

Every compute step runs in the library's CUDA kernels; this module checks
tensor dtypes/devices, allocates outputs with torch when the caller gives
none, and forwards raw device pointers plus the current CUDA stream.  There
is no fallback: if the library is missing or a call fails, it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoedec.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_ARG", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_LIMIT",
                -4: "MOE_ERR_WORKSPACE", -5: "MOE_ERR_ALIGN", -6: "MOE_ERR_CUDA",
                -7: "MOE_ERR_DEVICE"}

# every symbol include/moedec.h declares
EXPORTS = ("moe_version", "moe_strerror", "moe_gate_up", "moe_down", "moe_layer_workspace_bytes",
           "moe_layer", "moe_layer_host_workspace_bytes", "moe_layer_host", "moe_align_sizes",
           "moe_align_block_size", "moe_align_block_size_static", "moe_align_static_fits",
           "moe_copy", "moe_device_error", "moe_router_topk", "moe_mx_requant", "moe_gate_up_fp4",
           "moe_layer_grouped_workspace_bytes", "moe_layer_grouped",
           "moe_down_fp4")


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)} ({msg})")
        self.status = status


class MXView(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("s", ctypes.c_void_p)]


class MX(NamedTuple):
    """MXFP8 tensor: codes uint8 [E, rows, K] and E8M0 scales uint8 [E, rows, K/32]."""
    w: torch.Tensor
    s: torch.Tensor


_lib = None


def load(path: str = LIB_PATH):
    """Load libmoedec.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoedec.so not found at {path}: build it first "
                           "(python -m mixture_experts_decode_gb300.build)")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    MXP = ctypes.POINTER(MXView)
    sig = {
        "moe_version": ([], I),
        "moe_strerror": ([I], ctypes.c_char_p),
        "moe_gate_up": ([P, I, I, P, I, MXView, MXView, I, I, MXP, MXP, P, P], I),
        "moe_down": ([P, I, I, P, P, MXView, I, I, I, MXP, P, P], I),
        "moe_layer_workspace_bytes": ([I, I, I, I, ctypes.POINTER(S)], I),
        "moe_layer": ([P, I, I, P, P, I, MXView, MXView, MXView, I, I, MXP, MXP, MXP, P, S, P, P], I),
        "moe_layer_host_workspace_bytes": ([I, I, I, I, I, ctypes.POINTER(S)], I),
        "moe_layer_host": ([P, I, I, P, P, I, MXView, MXView, MXView, I, I, MXP, MXP, MXP, P, S, P, P], I),
        "moe_align_sizes": ([I, I, I, I, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                             ctypes.POINTER(S)], I),
        "moe_align_block_size": ([P, I, I, I, I, P, P, P, P, S, P], I),
        "moe_router_topk": ([P, I, I, I, I, ctypes.c_float, P, P, P], I),
        "moe_mx_requant": ([P, P, ctypes.c_int64, I, P], I),
        "moe_gate_up_fp4": ([P, I, I, P, I, MXView, MXView, I, I, MXP, MXP, P, P], I),
        "moe_down_fp4": ([P, I, I, P, P, MXView, I, I, I, MXP, P, P], I),
        "moe_align_block_size_static": ([P, I, I, I, I, P, P, P, P], I),
        "moe_align_static_fits": ([I, I, I], I),
        "moe_copy": ([P, P, S, P], I),
        "moe_device_error": ([P, ctypes.POINTER(I)], I),
        "moe_layer_grouped_workspace_bytes": ([I, I, I, I, I, I, ctypes.POINTER(S)], I),
        "moe_layer_grouped": ([P, I, I, P, P, I, MXView, MXView, MXView, I, I, MXP, MXP, MXP, I, P, S, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoEError(fn, rc, load().moe_strerror(rc).decode())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _mx(m: Optional[MX], name: str, device, rows: int, K: int, E: Optional[int] = None, fp4: bool = False):
    if m is None:
        return None
    _need(m.w, name + ".w", torch.uint8, device, 3)
    _need(m.s, name + ".s", torch.uint8, device, 3)
    e = m.w.shape[0] if E is None else E
    kc = K // 2 if fp4 else K   # code bytes per row (MXFP4: two codes per byte)
    if tuple(m.w.shape) != (e, rows, kc) or tuple(m.s.shape) != (e, rows, K // 32):
        raise ValueError(f"{name}: expected codes [{e},{rows},{kc}] and scales [{e},{rows},{K // 32}], "
                         f"got {tuple(m.w.shape)} / {tuple(m.s.shape)}")
    return MXView(m.w.data_ptr(), m.s.data_ptr())


def _ref(v):
    return None if v is None else ctypes.byref(v)


def version() -> int:
    return load().moe_version()


def gate_up(x, topk_ids, w_gate: MX, w_up: MX, shared_gate: Optional[MX] = None,
            shared_up: Optional[MX] = None, h: Optional[torch.Tensor] = None, fp4: bool = False):
    """Fused gate/up pass; returns h BF16 [B, k+S, I].  fp4=True: MXFP4
    weights (codes [E, I, d/2], two E2M1 codes per byte) through
    moe_gate_up_fp4."""
    lib = load()
    dev = x.device
    _need(x, "x", torch.bfloat16, None, 2)
    _need(topk_ids, "topk_ids", torch.int32, dev, 2)
    B, d = x.shape
    k = topk_ids.shape[1]
    E, I = w_gate.w.shape[0], w_gate.w.shape[1]
    vg, vu = _mx(w_gate, "w_gate", dev, I, d, None, fp4), _mx(w_up, "w_up", dev, I, d, E, fp4)
    sg = _mx(shared_gate, "shared_gate", dev, I, d, 1, fp4)
    su = _mx(shared_up, "shared_up", dev, I, d, 1, fp4)
    S = 1 if sg is not None else 0
    if h is None:
        h = torch.empty((B, k + S, I), dtype=torch.bfloat16, device=dev)
    _need(h, "h", torch.bfloat16, dev)
    if h.numel() != B * (k + S) * I:
        raise ValueError("h has the wrong size")
    name = "moe_gate_up_fp4" if fp4 else "moe_gate_up"
    _check(name, getattr(lib, name)(x.data_ptr(), B, d, topk_ids.data_ptr(), k, vg, vu, E, I,
                                    _ref(sg), _ref(su), h.data_ptr(), _stream(dev)))
    return h


def down(h, topk_ids, topk_w, w_down: MX, shared_down: Optional[MX] = None,
         y: Optional[torch.Tensor] = None, fp4: bool = False):
    """Down pass with the routing-weighted combine folded in; returns y BF16
    [B, d].  fp4=True: MXFP4 weights (codes [E, d, I/2]) through moe_down_fp4."""
    lib = load()
    dev = h.device
    _need(h, "h", torch.bfloat16, None, 3)
    _need(topk_ids, "topk_ids", torch.int32, dev, 2)
    _need(topk_w, "topk_w", torch.float32, dev, 2)
    B, KS, I = h.shape
    k = topk_ids.shape[1]
    E, d = w_down.w.shape[0], w_down.w.shape[1]
    vd = _mx(w_down, "w_down", dev, d, I, None, fp4)
    sd = _mx(shared_down, "shared_down", dev, d, I, 1, fp4)
    if KS != k + (1 if sd is not None else 0):
        raise ValueError("h's middle dimension must be k (+1 with a shared expert)")
    if y is None:
        y = torch.empty((B, d), dtype=torch.bfloat16, device=dev)
    _need(y, "y", torch.bfloat16, dev)
    name = "moe_down_fp4" if fp4 else "moe_down"
    _check(name, getattr(lib, name)(h.data_ptr(), B, k, topk_ids.data_ptr(), topk_w.data_ptr(), vd,
                                    E, d, I, _ref(sd), y.data_ptr(), _stream(dev)))
    return y


def layer_workspace_bytes(B: int, k: int, I: int, has_shared: bool) -> int:
    out = ctypes.c_size_t()
    _check("moe_layer_workspace_bytes",
           load().moe_layer_workspace_bytes(B, k, I, int(has_shared), ctypes.byref(out)))
    return out.value


def _shared3(shared):
    if shared is None:
        return None, None, None
    if len(shared) != 3:
        raise ValueError("shared must be (gate, up, down) MX triples")
    return shared


def layer(x, topk_ids, topk_w, w_gate: MX, w_up: MX, w_down: MX, shared=None,
          workspace: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None):
    """The whole decode layer (gate/up then down on the current stream)."""
    lib = load()
    dev = x.device
    _need(x, "x", torch.bfloat16, None, 2)
    _need(topk_ids, "topk_ids", torch.int32, dev, 2)
    _need(topk_w, "topk_w", torch.float32, dev, 2)
    B, d = x.shape
    k = topk_ids.shape[1]
    E, I = w_gate.w.shape[0], w_gate.w.shape[1]
    sg, su, sd = _shared3(shared)
    vg, vu = _mx(w_gate, "w_gate", dev, I, d), _mx(w_up, "w_up", dev, I, d, E)
    vd = _mx(w_down, "w_down", dev, d, I, E)
    vsg, vsu, vsd = (_mx(sg, "shared_gate", dev, I, d, 1), _mx(su, "shared_up", dev, I, d, 1),
                     _mx(sd, "shared_down", dev, d, I, 1))
    need = layer_workspace_bytes(B, k, I, shared is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if y is None:
        y = torch.empty((B, d), dtype=torch.bfloat16, device=dev)
    _need(y, "y", torch.bfloat16, dev)
    _check("moe_layer", lib.moe_layer(x.data_ptr(), B, d, topk_ids.data_ptr(), topk_w.data_ptr(), k,
                                      vg, vu, vd, E, I, _ref(vsg), _ref(vsu), _ref(vsd),
                                      workspace.data_ptr(), workspace.numel(), y.data_ptr(),
                                      _stream(dev)))
    return y


def layer_grouped_workspace_bytes(T: int, k: int, E: int, d: int, I: int, has_shared: bool = False) -> int:
    out = ctypes.c_size_t()
    _check("moe_layer_grouped_workspace_bytes",
           load().moe_layer_grouped_workspace_bytes(T, k, E, d, I, int(has_shared), ctypes.byref(out)))
    return out.value


def layer_grouped(x, topk_ids, topk_w, w_gate: MX, w_up: MX, w_down: MX, shared=None, act_mx: bool = False,
                  workspace: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None):
    """The layer computed expert-centrically (align, grouped tensor-core GEMMs,
    combine) on the current stream; act_mx rounds x and h through MXFP8;
    shared = (gate, up, down) MX triples of a shared expert, or None."""
    lib = load()
    dev = x.device
    _need(x, "x", torch.bfloat16, None, 2)
    _need(topk_ids, "topk_ids", torch.int32, dev, 2)
    _need(topk_w, "topk_w", torch.float32, dev, 2)
    T, d = x.shape
    k = topk_ids.shape[1]
    E, I = w_gate.w.shape[0], w_gate.w.shape[1]
    vg, vu = _mx(w_gate, "w_gate", dev, I, d), _mx(w_up, "w_up", dev, I, d, E)
    vd = _mx(w_down, "w_down", dev, d, I, E)
    sg, su, sd = _shared3(shared)
    vsg, vsu, vsd = (_mx(sg, "shared_gate", dev, I, d, 1), _mx(su, "shared_up", dev, I, d, 1),
                     _mx(sd, "shared_down", dev, d, I, 1))
    need = layer_grouped_workspace_bytes(T, k, E, d, I, shared is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    _need(y, "y", torch.bfloat16, dev)
    _check("moe_layer_grouped", lib.moe_layer_grouped(
        x.data_ptr(), T, d, topk_ids.data_ptr(), topk_w.data_ptr(), k, vg, vu, vd, E, I, _ref(vsg), _ref(vsu),
        _ref(vsd), int(bool(act_mx)), workspace.data_ptr(), workspace.numel(), y.data_ptr(), _stream(dev)))
    return y


def layer_host_workspace_bytes(B: int, d: int, k: int, I: int, has_shared: bool) -> int:
    out = ctypes.c_size_t()
    _check("moe_layer_host_workspace_bytes",
           load().moe_layer_host_workspace_bytes(B, d, k, I, int(has_shared), ctypes.byref(out)))
    return out.value


def layer_host(x_host, topk_ids_host, topk_w_host, w_gate: MX, w_up: MX, w_down: MX, shared=None,
               workspace: Optional[torch.Tensor] = None, y_host: Optional[torch.Tensor] = None,
               device=None):
    """moe_layer_host: activations in (pinned) host memory, weights on the GPU.

    Asynchronous on the current stream of the weights' device; synchronise
    before reading y_host."""
    lib = load()
    dev = device or w_gate.w.device
    _need(x_host, "x_host", torch.bfloat16, torch.device("cpu"), 2)
    _need(topk_ids_host, "topk_ids_host", torch.int32, torch.device("cpu"), 2)
    _need(topk_w_host, "topk_w_host", torch.float32, torch.device("cpu"), 2)
    B, d = x_host.shape
    k = topk_ids_host.shape[1]
    E, I = w_gate.w.shape[0], w_gate.w.shape[1]
    sg, su, sd = _shared3(shared)
    vg, vu = _mx(w_gate, "w_gate", dev, I, d), _mx(w_up, "w_up", dev, I, d, E)
    vd = _mx(w_down, "w_down", dev, d, I, E)
    vsg, vsu, vsd = (_mx(sg, "shared_gate", dev, I, d, 1), _mx(su, "shared_up", dev, I, d, 1),
                     _mx(sd, "shared_down", dev, d, I, 1))
    need = layer_host_workspace_bytes(B, d, k, I, shared is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if y_host is None:
        y_host = torch.empty((B, d), dtype=torch.bfloat16).pin_memory()
    _need(y_host, "y_host", torch.bfloat16, torch.device("cpu"), 2)
    _check("moe_layer_host", lib.moe_layer_host(
        x_host.data_ptr(), B, d, topk_ids_host.data_ptr(), topk_w_host.data_ptr(), k, vg, vu, vd, E, I,
        _ref(vsg), _ref(vsu), _ref(vsd), workspace.data_ptr(), workspace.numel(), y_host.data_ptr(),
        _stream(dev)))
    return y_host


def align_sizes(T: int, k: int, E: int, block_size: int):
    """(n_sorted, n_blocks, workspace_bytes) for align_block_size."""
    ns, nb, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    _check("moe_align_sizes", load().moe_align_sizes(T, k, E, block_size, ctypes.byref(ns),
                                                      ctypes.byref(nb), ctypes.byref(ws)))
    return ns.value, nb.value, ws.value


def align_block_size(topk_ids, E: int, block_size: int, sorted_token_ids=None, expert_ids=None,
                     num_tokens_post_pad=None, workspace=None):
    """moe_align_block_size; returns (sorted_token_ids, expert_ids, num_tokens_post_pad)."""
    lib = load()
    dev = topk_ids.device
    _need(topk_ids, "topk_ids", torch.int32, None, 2)
    T, k = topk_ids.shape
    ns, nb, wsb = align_sizes(T, k, E, block_size)
    if sorted_token_ids is None:
        sorted_token_ids = torch.empty(ns, dtype=torch.int32, device=dev)
    if expert_ids is None:
        expert_ids = torch.empty(nb, dtype=torch.int32, device=dev)
    if num_tokens_post_pad is None:
        num_tokens_post_pad = torch.empty(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    for t, nm in ((sorted_token_ids, "sorted_token_ids"), (expert_ids, "expert_ids"),
                  (num_tokens_post_pad, "num_tokens_post_pad")):
        _need(t, nm, torch.int32, dev)
    if sorted_token_ids.numel() < ns or expert_ids.numel() < nb:
        raise ValueError("align output buffers are too small")
    _check("moe_align_block_size", lib.moe_align_block_size(
        topk_ids.data_ptr(), T, k, E, block_size, sorted_token_ids.data_ptr(), expert_ids.data_ptr(),
        num_tokens_post_pad.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(dev)))
    return sorted_token_ids, expert_ids, num_tokens_post_pad


def align_block_size_static(topk_ids, E: int, block_size: int, sorted_token_ids=None,
                            expert_ids=None, num_tokens_post_pad=None):
    """moe_align_block_size_static: the same result with the library's fixed
    scratch array instead of a caller workspace (see include/moedec.h)."""
    lib = load()
    dev = topk_ids.device
    _need(topk_ids, "topk_ids", torch.int32, None, 2)
    T, k = topk_ids.shape
    ns, nb, _ = align_sizes(T, k, E, block_size)
    if sorted_token_ids is None:
        sorted_token_ids = torch.empty(ns, dtype=torch.int32, device=dev)
    if expert_ids is None:
        expert_ids = torch.empty(nb, dtype=torch.int32, device=dev)
    if num_tokens_post_pad is None:
        num_tokens_post_pad = torch.empty(1, dtype=torch.int32, device=dev)
    _check("moe_align_block_size_static", lib.moe_align_block_size_static(
        topk_ids.data_ptr(), T, k, E, block_size, sorted_token_ids.data_ptr(), expert_ids.data_ptr(),
        num_tokens_post_pad.data_ptr(), _stream(dev)))
    return sorted_token_ids, expert_ids, num_tokens_post_pad


def copy(dst: torch.Tensor, src: torch.Tensor):
    """The library's bandwidth-reference copy kernel (bytes = src.nbytes)."""
    if dst.nbytes < src.nbytes:
        raise ValueError("dst smaller than src")
    _check("moe_copy", load().moe_copy(dst.data_ptr(), src.data_ptr(), src.nbytes, _stream(src.device)))
    return dst


def device_error(device=None) -> int:
    """Synchronise the current stream; return and clear the device error bits."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    bits = ctypes.c_int()
    rc = load().moe_device_error(_stream(dev), ctypes.byref(bits))
    if rc not in (MOE_OK, -7):
        _check("moe_device_error", rc)
    return bits.value


ROUTER_SCORES = {"softmax": 0, "sigmoid": 1}


def router_topk(logits, k: int, score: str = "softmax", scale: float = 1.0, topk_ids=None, topk_w=None):
    """moe_router_topk: logits float32 [B, E] (device) -> (topk_ids int32 [B, k],
    topk_w float32 [B, k]); score "softmax" (renormalised top-k) or "sigmoid"
    (normalised over the k, times `scale`)."""
    lib = load()
    dev = logits.device
    _need(logits, "logits", torch.float32, None, 2)
    B, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((B, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((B, k), dtype=torch.float32, device=dev)
    _need(topk_ids, "topk_ids", torch.int32, dev)
    _need(topk_w, "topk_w", torch.float32, dev)
    _check("moe_router_topk", lib.moe_router_topk(logits.data_ptr(), B, E, k, ROUTER_SCORES[score], float(scale),
                                                  topk_ids.data_ptr(), topk_w.data_ptr(), _stream(dev)))
    return topk_ids, topk_w


def mx_requant(x, out=None):
    """moe_mx_requant: BF16 [..., K] (device, contiguous, K % 32 == 0) ->
    the same values through MXFP8 (OCP MX v1.0, blocks of 32 along the last
    axis) and back to BF16.  out may be x itself."""
    lib = load()
    _need(x, "x", torch.bfloat16)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, x.device)
    if out.shape != x.shape:
        raise ValueError("out must have the shape of x")
    K = x.shape[-1] if x.dim() else 0
    rows = x.numel() // K if K else 0
    _check("moe_mx_requant", lib.moe_mx_requant(x.data_ptr(), out.data_ptr(), rows, K, _stream(x.device)))
    return out
