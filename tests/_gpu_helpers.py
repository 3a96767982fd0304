"""Shared helpers of the GPU parity tests (not collected by pytest)."""
from __future__ import annotations

import os

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


def oracle_tokens(W, x, ids, w, tokens, mx_act=False):
    """Oracle layer for a subset of tokens, passing only the experts they touch
    (mx_act: the variant with x and h rounded through MXFP8)."""
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
    fn = oracle.moe_layer_mx_act if mx_act else oracle.moe_layer
    return fn(bf16_bits(x[tokens]), remap[sub_ids].astype(np.int32), w[tokens].cpu().numpy(), *host,
              shared=shared)


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


def h_interval(ref, abs_g, abs_u, eps_ulps=EPS_ULPS):
    """Bounds (lo, hi) of the exact h that an FP32 evaluation may have seen
    (dot products within eps_ulps units of 2^-24 of sum |x * w|)."""
    g, u, h = ref["g64"], ref["u64"], ref["h64"]
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    eg = eps_ulps * 2.0 ** -24 * abs_g
    eu = eps_ulps * 2.0 ** -24 * abs_u
    dh = np.abs(dsilu * u) * eg + np.abs(_silu(g)) * eu + eg * eu + 8 * 2.0 ** -24 * np.abs(h)
    return h - dh, h + dh


def abs_matrix(W, which: str, e: int) -> torch.Tensor:
    """|dequantised weight matrix| of expert e (e < 0: the shared expert), FP32
    on the CPU (exact for these weights; it only feeds error bounds)."""
    if e < 0:
        i = {"gate": 0, "up": 2, "down": 4}[which]
        codes, scales = W["shared"][i][0], W["shared"][i + 1][0]
    else:
        codes, scales = W["w_" + which][e], W["s_" + which][e]
    rows, K = codes.shape
    c = codes.cpu().contiguous().view(torch.float8_e4m3fn).to(torch.float32).abs()
    sc = torch.exp2(scales.cpu().to(torch.float32) - 127.0)
    return (c.view(rows, K // 32, 32) * sc.view(rows, K // 32, 1)).view(rows, K)


def _slot_expert(ids_tok, b, j, k):
    return int(ids_tok[b, j]) if j < k else -1


def _slots_by_expert(ids_tok, KS):
    """{expert: [(b, j), ...]} over every slot (j == k is the shared expert, -1)."""
    T, k = ids_tok.shape
    out = {}
    for b in range(T):
        for j in range(KS):
            out.setdefault(_slot_expert(ids_tok, b, j, k), []).append((b, j))
    return out


def abs_sums(W, x_tok, ids_tok, KS):
    """sum_c |x_c * Wg[n, c]| and the same for Wu, per (token, slot, neuron);
    one expert's matrices at a time."""
    T = ids_tok.shape[0]
    ax = torch.from_numpy(np.abs(x_tok)).to(torch.float32)
    sg = su = None
    for e, slots in _slots_by_expert(ids_tok, KS).items():
        bs = [b for b, _ in slots]
        g = (abs_matrix(W, "gate", e) @ ax[bs].T).T.double().numpy()
        u = (abs_matrix(W, "up", e) @ ax[bs].T).T.double().numpy()
        if sg is None:
            sg = np.zeros((T, KS, g.shape[1]))
            su = np.zeros_like(sg)
        for i, (b, j) in enumerate(slots):
            sg[b, j], su[b, j] = g[i], u[i]
    return sg, su


def tc_y_allowance(W, ids_tok, w_tok, ref, x_tok, d, K_gu, K_dn):
    """Allowance for a layer whose dot products are summed by the tensor
    cores in FP32 (K / 16 MMA steps, each adding a 16-product partial): the
    standard bound of recursive FP32 summation, (steps + 16) units of 2^-24
    of the sum of the terms' magnitudes, per dot product.  Gate/up: every h
    whose interval under that bound holds two BF16 roundings moves y by
    sum_j |w_j| sum_i |Wd| * (round(hi) - round(lo)); down: each slot's row
    may be off by (K_dn / 16 + 16) units of sum_i |h Wd|, times |w_j|, and
    the combine's k + 1 additions a few units more.  Computed from the
    oracle's values and the weights only."""
    KS = ref["h"].shape[1]
    k = ids_tok.shape[1]
    ag, au = abs_sums(W, x_tok, ids_tok, KS)
    lo, hi = h_interval(ref, ag, au, eps_ulps=K_gu / 16 + 16)
    gap = _bf16_value(_bf16_round_vec(hi)) - _bf16_value(_bf16_round_vec(lo))
    allow = y_allowance(W, ids_tok, w_tok, gap, d) if np.any(gap) else np.zeros((ids_tok.shape[0], d))
    # the down products and the combine
    habs = np.abs(_bf16_value(ref["h"]))
    T = ids_tok.shape[0]
    acc = np.zeros((T, d))
    for e, slots in _slots_by_expert(ids_tok, KS).items():
        A = abs_matrix(W, "down", e)
        for b, j in slots:
            wt = abs(float(w_tok[b, j])) if j < k else 1.0
            acc[b] += wt * (A @ torch.from_numpy(habs[b, j]).to(torch.float32)).double().numpy()
    return allow + (K_dn / 16 + 16 + k + 1) * 2.0 ** -24 * acc, int(np.count_nonzero(gap))


def y_allowance(W, ids_tok, w_tok, gap, d):
    """Per-output allowance for the h whose BF16 rounding is not unique."""
    T, KS, I = gap.shape
    k = ids_tok.shape[1]
    allow = np.zeros((T, d))
    for e, slots in _slots_by_expert(ids_tok, KS).items():
        slots = [(b, j) for b, j in slots if np.any(gap[b, j])]
        if not slots:
            continue
        A = abs_matrix(W, "down", e)
        for b, j in slots:
            wt = abs(float(w_tok[b, j])) if j < k else 1.0
            allow[b] += wt * (A @ torch.from_numpy(gap[b, j]).to(torch.float32)).double().numpy()
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


def check_plain(got: torch.Tensor, ref64: np.ndarray, what: str, allow=None) -> float:
    """The plain bar |gpu - y64| <= TOL * max(1, |y64|), plus `allow` where
    given (the effect of h values the GPU rounded the other valid way)."""
    g = got.detach().float().cpu().double().numpy().reshape(ref64.shape)
    err = np.abs(g - ref64)
    scaled = err / np.maximum(1.0, np.abs(ref64))
    worst = float(scaled.max()) if scaled.size else 0.0
    if allow is None:
        assert worst <= TOL, f"{what}: max plain scaled error {worst:.3e} > {TOL}"
    else:
        excess = (np.maximum(err - allow, 0.0) / np.maximum(1.0, np.abs(ref64))).max()
        assert excess <= TOL, (f"{what}: max scaled error beyond the rounding differences of h "
                               f"{excess:.3e} > {TOL} (plain {worst:.3e})")
    return worst


def _report(line: str):
    path = os.environ.get("MOEDEC_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def compare_tokens(dev, W, Wd, x, ids, w, tokens, what, chunk=8, plain=True):
    """GPU layer on the whole batch vs the oracle on `tokens` (in chunks of
    `chunk` tokens, so only their experts are held on the host); checks h
    (valid BF16 rounding), y against the tolerance with the rounding
    allowance, y against the plain tolerance, and the per-token cosine.

    plain=False (layers whose y reach |y| > 1, where BF16 rounding of y alone
    may take 3.906e-3 of the 4e-3): y must meet the plain tolerance plus the
    exact effect of the h values where the GPU's BF16 rounding differs from
    the oracle's (both valid: the exact h lies within FP32 error of a BF16
    midpoint), i.e. sum_j |w_j| sum_i |Wd[e_j, o, i]| |h_gpu - h_oracle|_i;
    with no such h it is the plain bar itself."""
    y = run_layer(dev, Wd, x, ids, w)
    h = run_gate_up(dev, Wd, x, ids)
    torch.cuda.synchronize()
    assert moe.device_error(dev) == 0
    tokens = list(tokens)
    d = y.shape[1]
    n_gap, n_diff, worst, worst_plain, cos_min = 0, 0, 0.0, 0.0, 1.0
    for c0 in range(0, len(tokens), chunk):
        toks = tokens[c0:c0 + chunk]
        ref = oracle_tokens(W, x, ids, w, toks)
        t = torch.tensor(toks, dtype=torch.long, device=dev)
        ids_tok, w_tok = ids[toks].cpu().numpy(), w[toks].cpu().numpy()
        x_tok = x[toks].float().double().numpy()
        KS = ref["h"].shape[1]
        ag, au = abs_sums(W, x_tok, ids_tok, KS)
        lo, hi = h_interval(ref, ag, au)
        ht = h.index_select(0, t)
        gap = check_h(ht, ref, lo, hi, what + " h")
        allow = y_allowance(W, ids_tok, w_tok, gap, d) if np.any(gap) else None
        yt = y.index_select(0, t)
        worst = max(worst, check_close(yt, ref["y64"], what + " y", allow))
        diff = np.abs(_bf16_value(bf16_bits(ht).reshape(ref["h"].shape)) - _bf16_value(ref["h"]))
        n_diff += int(np.count_nonzero(diff))
        obs = None
        if not plain and np.any(diff):
            obs = y_allowance(W, ids_tok, w_tok, diff, d)
        worst_plain = max(worst_plain, check_plain(yt, ref["y64"], what + " y", None if plain else obs))
        cos_min = min(cos_min, check_cosine(yt, ref["y64"], what + " y"))
        n_gap += int(np.count_nonzero(gap))
    _report(f"{what}: tokens {len(tokens)}/{x.shape[0]}, max plain scaled error {worst_plain:.3e} "
            f"({'asserted' if plain else 'asserted beyond the observed h rounding differences'}), "
            f"with allowance {worst:.3e}, min cosine {cos_min:.8f}, h with two valid roundings {n_gap}, "
            f"h rounded the other valid way {n_diff}")
    return n_gap, worst_plain, cos_min


def item_cover(ids, shared: bool, tc: int = 4):
    """Tokens such that every work item of the decode passes, (expert, group
    of tc of its tokens in increasing order), holds at least one of them:
    a greedy set cover."""
    ids = np.asarray(ids)
    B = ids.shape[0]
    groups = []
    for e in sorted(set(ids.reshape(-1).tolist())):
        toks = sorted(set(np.nonzero((ids == e).any(1))[0].tolist()))
        groups += [set(toks[i:i + tc]) for i in range(0, len(toks), tc)]
    if shared:
        groups += [set(range(i, min(B, i + tc))) for i in range(0, B, tc)]
    chosen = set()
    left = [g for g in groups]
    while left:
        counts = {}
        for g in left:
            for b in g:
                counts[b] = counts.get(b, 0) + 1
        best = min(counts, key=lambda b: (-counts[b], b))
        chosen.add(best)
        left = [g for g in left if best not in g]
    return sorted(chosen)


def small_weights(E, d, I, shared, seed, dev="cpu"):
    cfg = inputs.LayerConfig(f"edge_{E}_{d}_{I}_{int(shared)}_{seed}", E, 1, d, I, shared, "softmax_normal")
    return inputs.layer_weights(cfg, dev)
