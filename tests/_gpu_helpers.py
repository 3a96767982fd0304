"""Shared helpers of the GPU parity tests (not collected by pytest)."""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_decode_gb300 as moe
import oracle
from mixture_experts_decode_gb300 import inputs

# Acceptance rule of the decode layer, per output element:
#   |gpu - oracle| <= 4e-3 * max(1, |oracle|)   and per-token cosine >= 0.99999,
# against the oracle's UNROUNDED FP64 value.  BF16 round-to-nearest alone
# contributes at most 2^-8 * |v| (< 3.91e-3 |v|), leaving ~9e-5 |v| for FP32
# accumulation-order differences.
TOL = 4e-3
COS = 0.99999
# The intermediate h is BF16, rounded from an FP32 value.  An FP32 dot
# product's error is bounded relative to the sum of the absolute values of
# its terms, not to the result, so: with S = sum_c |x_c * w_c| for the gate
# and the up dot, each may be off by EPS_ULPS * 2^-24 * S; propagated through
# SiLU(g) * u (plus a few FP32 ulps for SiLU itself) this gives an interval
# around the exact h.  Every BF16 value the interval's ends round to (and any
# between) is a correct h: GPU h must lie within [round(lo), round(hi)], which
# for most h is the oracle's value itself, bit for bit.  y then gets an
# allowance of sum_j |w_j| * sum_i |Wd[e_j, o, i]| * (round(hi) - round(lo))_i
# on top of TOL.  All of it comes from the oracle's values and the weights.
EPS_ULPS = 4.0

WEIGHT_NAMES = ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def device_mx(W, dev):
    mx = lambda a, b: moe.MX(W[a].to(dev), W[b].to(dev))
    out = dict(gate=mx("w_gate", "s_gate"), up=mx("w_up", "s_up"), down=mx("w_down", "s_down"))
    shared = None
    if W.get("shared") is not None:
        s = [t.to(dev) for t in W["shared"]]
        shared = (moe.MX(s[0], s[1]), moe.MX(s[2], s[3]), moe.MX(s[4], s[5]))
    out["shared"] = shared
    return out


def oracle_tokens(W, x, ids, w, tokens):
    """Oracle layer for a subset of tokens, passing only the experts they touch."""
    tokens = list(tokens)
    sub_ids = ids[tokens].cpu().numpy()
    uniq = sorted(set(sub_ids.reshape(-1).tolist()))
    remap = np.full(max(uniq) + 1, -1, np.int64)
    remap[uniq] = np.arange(len(uniq))
    idx = torch.tensor(uniq, dtype=torch.long)
    host = [W[n].index_select(0, idx.to(W[n].device)).cpu().numpy() for n in WEIGHT_NAMES]
    shared = None
    if W.get("shared") is not None:
        shared = tuple(t.cpu().numpy() for t in W["shared"])
    return oracle.moe_layer(bf16_bits(x[tokens]), remap[sub_ids].astype(np.int32),
                            w[tokens].cpu().numpy(), *host, shared=shared)


def check_close(got: torch.Tensor, ref64: np.ndarray, what: str, allow=None):
    g = got.detach().float().cpu().double().numpy().reshape(ref64.shape)
    excess = np.abs(g - ref64) - (0.0 if allow is None else allow)
    scaled = np.maximum(excess, 0.0) / np.maximum(1.0, np.abs(ref64))
    worst = float(scaled.max()) if scaled.size else 0.0
    assert worst <= TOL, f"{what}: max scaled error {worst:.3e} > {TOL}"
    return worst


def check_cosine(got: torch.Tensor, ref64: np.ndarray, what: str):
    g = got.detach().float().cpu().double().numpy().reshape(ref64.shape)
    g2 = g.reshape(g.shape[0], -1)
    r2 = ref64.reshape(ref64.shape[0], -1)
    num = np.sum(g2 * r2, axis=1)
    den = np.linalg.norm(g2, axis=1) * np.linalg.norm(r2, axis=1)
    ok = den > 0
    cos = np.where(ok, num / np.where(ok, den, 1.0), 1.0)
    assert np.all(cos >= COS), f"{what}: min cosine {cos.min():.8f} < {COS}"
    # an all-zero reference must give an all-zero output
    assert np.all(np.abs(g2[~ok]) == 0) if np.any(~ok) else True
    return float(cos.min())


def _bf16_round_vec(v: np.ndarray) -> np.ndarray:
    flat = v.reshape(-1)
    out = np.fromiter((oracle.bf16_round(float(a)) for a in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(v.shape)


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _silu(g):
    return g / (1.0 + np.exp(-g))


def h_interval(ref, abs_g, abs_u):
    """Bounds (lo, hi) of the exact h that an FP32 evaluation may have seen."""
    g, u, h = ref["g64"], ref["u64"], ref["h64"]
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    eg = EPS_ULPS * 2.0 ** -24 * abs_g
    eu = EPS_ULPS * 2.0 ** -24 * abs_u
    dh = np.abs(dsilu * u) * eg + np.abs(_silu(g)) * eu + eg * eu + 8 * 2.0 ** -24 * np.abs(h)
    return h - dh, h + dh


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.ldexp(c, np.repeat(scales.astype(np.int64) - 127, 32, axis=-1))


class ExpertCache:
    """Dequantised (float64) expert matrices, fetched from the weight dict."""

    def __init__(self, W):
        self.W, self.c = W, {}

    def get(self, which: str, e: int):
        key = (which, e)
        if key not in self.c:
            if e < 0:       # the shared expert
                i = {"gate": 0, "up": 2, "down": 4}[which]
                codes, scales = self.W["shared"][i][0], self.W["shared"][i + 1][0]
            else:
                codes, scales = self.W["w_" + which][e], self.W["s_" + which][e]
            self.c[key] = dequant(codes.cpu().numpy(), scales.cpu().numpy())
        return self.c[key]


def _slot_expert(ids_tok, b, j, k):
    return int(ids_tok[b, j]) if j < k else -1


def abs_sums(cache, x_tok, ids_tok, KS):
    """sum_c |x_c * Wg[n, c]| and the same for Wu, per (token, slot, neuron)."""
    T, k = ids_tok.shape
    ax = np.abs(x_tok)
    sg, su = [], []
    for b in range(T):
        rg, ru = [], []
        for j in range(KS):
            e = _slot_expert(ids_tok, b, j, k)
            rg.append(np.abs(cache.get("gate", e)) @ ax[b])
            ru.append(np.abs(cache.get("up", e)) @ ax[b])
        sg.append(rg)
        su.append(ru)
    return np.array(sg), np.array(su)


def y_allowance(cache, ids_tok, w_tok, gap):
    """Per-output allowance for the h whose BF16 rounding is not unique."""
    T, KS, I = gap.shape
    k = ids_tok.shape[1]
    d = cache.get("down", _slot_expert(ids_tok, 0, 0, k)).shape[0]
    allow = np.zeros((T, d))
    for b in range(T):
        for j in range(KS):
            if not np.any(gap[b, j]):
                continue
            e = _slot_expert(ids_tok, b, j, k)
            wt = abs(float(w_tok[b, j])) if j < k else 1.0
            allow[b] += wt * (np.abs(cache.get("down", e)) @ gap[b, j])
    return allow


def check_h(h_gpu: torch.Tensor, ref, lo, hi, what: str):
    """h must be a correct BF16 rounding: within [round(lo), round(hi)]."""
    got = _bf16_value(bf16_bits(h_gpu).reshape(ref["h"].shape))
    rlo = _bf16_value(_bf16_round_vec(lo))
    rhi = _bf16_value(_bf16_round_vec(hi))
    bad = (got < rlo) | (got > rhi)
    assert not np.any(bad), (f"{what}: {int(bad.sum())} h outside the valid roundings, e.g. "
                             f"got {got[bad][:4]} want [{rlo[bad][:4]}, {rhi[bad][:4]}]")
    firm = rlo == rhi
    assert np.array_equal(bf16_bits(h_gpu).reshape(ref["h"].shape)[firm], ref["h"][firm])
    check_close(h_gpu, ref["h64"], what)
    return rhi - rlo


def run_layer(dev, Wd, x, ids, w):
    return moe.layer(x.to(dev), ids.to(dev), w.to(dev), Wd["gate"], Wd["up"], Wd["down"],
                     shared=Wd["shared"])


def run_gate_up(dev, Wd, x, ids):
    sh = Wd["shared"]
    return moe.gate_up(x.to(dev), ids.to(dev), Wd["gate"], Wd["up"],
                       shared_gate=sh[0] if sh else None, shared_up=sh[1] if sh else None)


def compare_tokens(dev, W, Wd, x, ids, w, tokens, what):
    """GPU layer on the whole batch vs the oracle on `tokens`; checks h and y."""
    y = run_layer(dev, Wd, x, ids, w)
    h = run_gate_up(dev, Wd, x, ids)
    torch.cuda.synchronize()
    ref = oracle_tokens(W, x, ids, w, tokens)
    t = torch.tensor(list(tokens), dtype=torch.long, device=dev)
    toks = list(tokens)
    ids_tok, w_tok = ids[toks].cpu().numpy(), w[toks].cpu().numpy()
    x_tok = x[toks].float().double().numpy()
    cache = ExpertCache(W)
    KS = ref["h"].shape[1]
    ag, au = abs_sums(cache, x_tok, ids_tok, KS)
    lo, hi = h_interval(ref, ag, au)
    gap = check_h(h.index_select(0, t), ref, lo, hi, what + " h")
    allow = y_allowance(cache, ids_tok, w_tok, gap) if np.any(gap) else None
    e_y = check_close(y.index_select(0, t), ref["y64"], what + " y", allow)
    c = check_cosine(y.index_select(0, t), ref["y64"], what + " y")
    assert moe.device_error(dev) == 0
    return int(np.count_nonzero(gap)), e_y, c


def small_weights(E, d, I, shared, seed, dev="cpu"):
    cfg = inputs.LayerConfig(f"edge_{E}_{d}_{I}_{int(shared)}_{seed}", E, 1, d, I, shared, "softmax_normal")
    return inputs.layer_weights(cfg, dev)
