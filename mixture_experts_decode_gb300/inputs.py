"""Seeded synthetic inputs for the MoE decode layer and for align.

This module draws random numbers and packs them into the library's layouts;
it holds none of the layer's arithmetic.  Both the CUDA path (tests, bench)
and the CPU oracle consume exactly the bytes produced here.

Recipe (every tensor is seeded from a hash of (workload, tensor, expert)):
  * x        ~ N(0, 1), rounded to BF16 (round-to-nearest-even).
  * W        ~ N(0, 0.02), quantised to MXFP8 with `quantize_mx`: for each
              block of 32 consecutive values along K, X = floor(log2 amax) - 8
              (8 = the largest E4M3 exponent), clamped to [-127, 127]; scale
              byte = X + 127 (E8M0); element = E4M3 round-to-nearest-even of
              v / 2^X, saturated to +-448.  An all-zero block gets scale 127.
              (FP4 variant, `quantize_mx4`: MXFP4, X = floor(log2 amax) - 2,
              E2M1 nearest with ties to the even code, saturated to +-6, two
              codes per byte with the lower K index in the low nibble.)
  * routing  (B rows, top-k of E):
      softmax_uniform  logits ~ U[0, 1), softmax, top-k, renormalised
      softmax_normal   logits ~ N(0, 1), softmax, top-k, renormalised
      sigmoid_scaled   scores = sigmoid(N(0, 1)), top-k, w = 2.5 * s / sum(s)
      zipf             popularity p_e ~ rank_e^-1.2 over a seeded permutation
                       of ranks; k distinct experts per token by Gumbel-top-k
                       on log p; w = softmax of fresh N(0, 1) over the k
      contiguous       token b slot j -> expert (b*k + j) mod E; w as zipf
    Top-k ties go to the lower expert index (stable sort).
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch

E4M3_MAX = 448.0
E4M3_EMAX = 8          # floor(log2(448))
MX_BLOCK = 32
E2M1_MAX = 6.0
E2M1_EMAX = 2          # floor(log2(6))
# E2M1 magnitudes of codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6: the midpoints
# between neighbouring codes, and whether a tie there goes up (to the even code)
_E2M1_STEPS = ((0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False), (3.5, True), (5.0, False))


def seed_for(*parts) -> int:
    """Deterministic 63-bit seed from any printable key parts."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *key) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(*key))
    return g


def randn(shape, device, *key, std=1.0) -> torch.Tensor:
    t = torch.randn(shape, generator=_gen(device, *key), device=device, dtype=torch.float32)
    return t * std if std != 1.0 else t


# ----------------------------------------------------------------- MXFP8 ---

def quantize_mx(v: torch.Tensor):
    """float32 [..., K] -> (E4M3 codes uint8 [..., K], E8M0 scales uint8 [..., K/32])."""
    K = v.shape[-1]
    assert K % MX_BLOCK == 0, "K must be a multiple of 32"
    blocks = v.reshape(*v.shape[:-1], K // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=-1)
    _, expo = torch.frexp(amax)                 # amax = m * 2^expo, m in [0.5, 1)
    X = (expo.to(torch.int32) - 1 - E4M3_EMAX)
    X = torch.where(amax > 0, X, torch.zeros_like(X)).clamp(-127, 127)
    factor = torch.exp2(-X.to(torch.float64)).unsqueeze(-1)   # exact power of two
    scaled = (blocks.to(torch.float64) * factor).to(torch.float32)
    scaled = scaled.clamp(-E4M3_MAX, E4M3_MAX)
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(v.shape)
    scales = (X + 127).to(torch.uint8)
    return codes.contiguous(), scales.contiguous()


def quantize_mx4(v: torch.Tensor):
    """float32 [..., K] -> (MXFP4 codes uint8 [..., K/2]: two E2M1 codes per
    byte, the lower K index in the low nibble; E8M0 scales uint8 [..., K/32]).
    X = floor(log2 amax) - 2 per block of 32 (2 = the largest E2M1 exponent),
    clamped to [-127, 127]; element = E2M1 nearest v / 2^X, ties to the even
    code, saturated to +-6; an all-zero block gets scale 127."""
    K = v.shape[-1]
    assert K % MX_BLOCK == 0, "K must be a multiple of 32"
    blocks = v.reshape(*v.shape[:-1], K // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=-1)
    _, expo = torch.frexp(amax)
    X = (expo.to(torch.int32) - 1 - E2M1_EMAX)
    X = torch.where(amax > 0, X, torch.zeros_like(X)).clamp(-127, 127)
    scaled = blocks.to(torch.float64) * torch.exp2(-X.to(torch.float64)).unsqueeze(-1)
    a = scaled.abs().clamp(max=E2M1_MAX)
    code = torch.zeros_like(a, dtype=torch.int32)
    for t, up in _E2M1_STEPS:
        code += (a >= t if up else a > t).to(torch.int32)
    code = code | ((scaled < 0) & (code > 0)).to(torch.int32) << 3
    code = code.reshape(v.shape).to(torch.uint8)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), (X + 127).to(torch.uint8).contiguous()


def mx4_weights(E: int, rows: int, K: int, device, *key, std=0.02):
    """E experts of [rows, K] MXFP4 weights ([E, rows, K/2] code bytes)."""
    codes = torch.empty((E, rows, K // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((E, rows, K // MX_BLOCK), dtype=torch.uint8, device=device)
    for e in range(E):
        codes[e], scales[e] = quantize_mx4(randn((rows, K), device, *key, e, std=std))
    return codes, scales


def mx_weights(E: int, rows: int, K: int, device, *key, std=0.02):
    """E experts of [rows, K] MXFP8 weights, generated one expert at a time."""
    codes = torch.empty((E, rows, K), dtype=torch.uint8, device=device)
    scales = torch.empty((E, rows, K // MX_BLOCK), dtype=torch.uint8, device=device)
    for e in range(E):
        w = randn((rows, K), device, *key, e, std=std)
        codes[e], scales[e] = quantize_mx(w)
    return codes, scales


# --------------------------------------------------------------- routing ---

def _topk_stable(scores: torch.Tensor, k: int):
    order = torch.sort(scores, dim=-1, descending=True, stable=True).indices
    return order[..., :k]


def route(kind: str, B: int, E: int, k: int, *key):
    """Return (topk_ids int32 [B, k], topk_w float32 [B, k]) on the CPU."""
    dev = "cpu"
    if kind in ("softmax_uniform", "softmax_normal"):
        g = _gen(dev, *key, "logits")
        if kind == "softmax_uniform":
            logits = torch.rand((B, E), generator=g, dtype=torch.float64)
        else:
            logits = torch.randn((B, E), generator=g, dtype=torch.float64)
        p = torch.softmax(logits, dim=-1)
        ids = _topk_stable(p, k)
        pk = torch.gather(p, 1, ids)
        w = pk / pk.sum(dim=-1, keepdim=True)
    elif kind == "sigmoid_scaled":
        g = _gen(dev, *key, "logits")
        s = torch.sigmoid(torch.randn((B, E), generator=g, dtype=torch.float64))
        ids = _topk_stable(s, k)
        sk = torch.gather(s, 1, ids)
        w = 2.5 * sk / sk.sum(dim=-1, keepdim=True)
    elif kind in ("zipf", "contiguous"):
        if kind == "zipf":
            g = _gen(dev, *key, "rank")
            rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
            logp = -1.2 * torch.log(rank)
            gu = torch.rand((B, E), generator=_gen(dev, *key, "gumbel"), dtype=torch.float64)
            gumbel = -torch.log(-torch.log(gu.clamp_min(1e-300)))
            ids = _topk_stable(logp.unsqueeze(0) + gumbel, k)
        else:
            ids = (torch.arange(B).unsqueeze(1) * k + torch.arange(k).unsqueeze(0)) % E
        z = torch.randn((B, k), generator=_gen(dev, *key, "weights"), dtype=torch.float64)
        w = torch.softmax(z, dim=-1)
    else:
        raise ValueError(f"unknown routing {kind!r}")
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def router_logits(kind: str, B: int, E: int, *key) -> torch.Tensor:
    """Router logits float32 [B, E] (CPU) with the distributions of the
    routings above: U[0, 1) for "softmax_uniform", N(0, 1) for
    "softmax_normal" and "sigmoid_scaled"."""
    g = _gen("cpu", *key, "router_logits")
    if kind == "softmax_uniform":
        return torch.rand((B, E), generator=g, dtype=torch.float32)
    if kind in ("softmax_normal", "sigmoid_scaled"):
        return torch.randn((B, E), generator=g, dtype=torch.float32)
    raise ValueError(f"no router logits for routing {kind!r}")


# ------------------------------------------------------------- workloads ---

@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    E: int
    k: int
    d: int
    I: int
    shared: bool
    routing: str


TINY = LayerConfig("tiny_e8_k2_d256_i128", 8, 2, 256, 128, False, "softmax_normal")
QWEN3 = LayerConfig("qwen3_e128_k8_d2048_i768", 128, 8, 2048, 768, False, "softmax_uniform")
DEEPSEEK_V3 = LayerConfig("deepseekv3_e256_k8_d7168_i2048_shared1", 256, 8, 7168, 2048, True,
                          "sigmoid_scaled")
CONFIGS = {c.name: c for c in (TINY, QWEN3, DEEPSEEK_V3)}


def layer_weights(cfg: LayerConfig, device="cpu", replica: int = 0, fp4: bool = False):
    """All expert weights of a layer (plus the shared expert when present);
    fp4=True draws the same way and packs MXFP4 (quantize_mx4) instead."""
    key = (cfg.name, "replica", replica) + (("fp4",) if fp4 else ())
    gen = mx4_weights if fp4 else mx_weights
    wg, sg = gen(cfg.E, cfg.I, cfg.d, device, *key, "w_gate")
    wu, su = gen(cfg.E, cfg.I, cfg.d, device, *key, "w_up")
    wd, sd = gen(cfg.E, cfg.d, cfg.I, device, *key, "w_down")
    out = dict(w_gate=wg, s_gate=sg, w_up=wu, s_up=su, w_down=wd, s_down=sd, shared=None)
    if cfg.shared:
        shg, shsg = gen(1, cfg.I, cfg.d, device, *key, "shared_gate")
        shu, shsu = gen(1, cfg.I, cfg.d, device, *key, "shared_up")
        shd, shsd = gen(1, cfg.d, cfg.I, device, *key, "shared_down")
        out["shared"] = (shg, shsg, shu, shsu, shd, shsd)
    return out


def expert_weights(cfg: LayerConfig, experts, device="cpu", replica: int = 0):
    """The weights of the listed experts only, stacked in that order: the same
    bytes layer_weights(cfg, device, replica) holds for those experts."""
    key = (cfg.name, "replica", replica)
    out = {}
    for name, rows, K in (("gate", cfg.I, cfg.d), ("up", cfg.I, cfg.d), ("down", cfg.d, cfg.I)):
        codes, scales = [], []
        for e in experts:
            c, s = quantize_mx(randn((rows, K), device, *key, "w_" + name, e, std=0.02))
            codes.append(c)
            scales.append(s)
        out["w_" + name] = torch.stack(codes)
        out["s_" + name] = torch.stack(scales)
    return out


def layer_batch(cfg: LayerConfig, B: int, routing: str | None = None, step: int = 0):
    """(x bf16 [B, d], topk_ids int32 [B, k], topk_w float32 [B, k]) on the CPU."""
    routing = routing or cfg.routing
    x = randn((B, cfg.d), "cpu", cfg.name, "x", B, step).to(torch.bfloat16)
    ids, w = route(routing, B, cfg.E, cfg.k, cfg.name, routing, B, step)
    return x.contiguous(), ids, w


def align_ids(T: int, k: int, E: int, routing: str = "softmax_normal", step: int = 0):
    """topk_ids int32 [T, k] for the align workload."""
    ids, _ = route(routing, T, E, k, "align", T, k, E, routing, step)
    return ids


def unique_experts(topk_ids: torch.Tensor) -> int:
    return int(torch.unique(topk_ids).numel())
