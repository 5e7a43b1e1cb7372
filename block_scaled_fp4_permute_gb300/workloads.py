"""Seeded synthetic workloads for the SiTU routed-MoE expert layer.

This module is the one place both sides of a parity test take their inputs
from: it draws routing, activations and weights, and packs the weights into
the block-scaled storage formats the layer consumes.  It holds none of the
layer's own arithmetic (no dequantisation, GEMM, activation, permute or
MXFP8 activation quantisation); weight packing is data preparation, the way
a checkpoint arrives already quantised.

Shapes follow the Kimi-K3 geometry of the TokenSpeed SiTU page ("Supported
contract": 896 experts, hidden 3584, top-k 16, TP8 intermediate 384 with all
896 experts local, EP8 intermediate 3072 with 112 local experts at
local_expert_offset = ep_rank * 112).

Recipe (seed s; small draws from numpy PCG64 streams spawned from
``SeedSequence([s, stream])``; the large weight tensors from torch's
generator on the target device, so that the 2 GB weight sets of the Kimi-K3
shapes take seconds, not minutes):
  * routing: ``uniform`` -- K distinct global IDs per token by argsort of
    uniforms; ``zipf(s)`` -- a seeded permutation assigns ranks, p_e is
    proportional to (rank+1)^-s and K distinct IDs are drawn per token by
    Gumbel-top-k (sampling without replacement);
  * topk_weights: softmax over K N(0,1) logits;
  * hidden states: N(0,1) rounded to bf16;
  * weights: N(0, 0.02) packed to MXFP4 (E2M1 + UE8M0 per 32 along K, scale
    = smallest 2^e with amax*2^-e <= 6, elements round-to-nearest-even) or
    NVFP4 (E2M1 + E4M3 per 16 along K + fp32 global scale amax/(6*448) per
    expert and W1 half);
  * NVFP4 activations: per-token global scale amax_t/(6*448), E4M3 block
    scale per 16, E2M1 elements;
  * per-expert SiTU constants: gemm1_alpha (beta) ~ U(0.5,1.5), gemm1_beta
    (linear beta) ~ U(0, 0.1), g1_alphas, g1_alphas_up ~ U(0.9, 1.1).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

ACT_BF16, ACT_MXFP8, ACT_NVFP4 = 0, 1, 2
ACT_FN_SITU, ACT_FN_SWIGLU_BIAS = 0, 1      # FC1 activation kinds
W_MXFP4, W_NVFP4 = 0, 1

# The workload families; "tiny" is small enough for the oracle in
# milliseconds, the others are Kimi-K3 shapes.
CONFIGS = {
    "tiny": dict(T=16, H=256, I=128, E_total=8, E_loc=8, off=0, K=2, act=ACT_BF16, wt=W_MXFP4,
                 routing=("uniform",), params="unit"),
    "decode": dict(T=64, H=3584, I=384, E_total=896, E_loc=896, off=0, K=16, act=ACT_BF16,
                   wt=W_MXFP4, routing=("uniform",), params="k3_random"),
    "prefill_w4a8": dict(T=8192, H=3584, I=384, E_total=896, E_loc=896, off=0, K=16,
                         act=ACT_MXFP8, wt=W_MXFP4, routing=("zipf", 1.0), params="k3_random"),
    "ep_shard": dict(T=4096, H=3584, I=3072, E_total=896, E_loc=112, off=336, K=16,
                     act=ACT_BF16, wt=W_MXFP4, routing=("uniform",), params="k3_random"),
    "nvfp4": dict(T=256, H=3584, I=384, E_total=896, E_loc=896, off=0, K=16, act=ACT_NVFP4,
                  wt=W_NVFP4, routing=("zipf", 0.8), params="k3_random"),
}
NVFP4_T_SWEEP = (1, 256, 2048, 16384)

_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _np_rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def _torch_gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) & 0x7FFF_FFFF_FFFF)
    return g


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def routing(T: int, K: int, E_total: int, kind=("uniform",), seed: int = 0):
    """Global top-k expert IDs (int32 [T,K], distinct per token) and fp32
    softmax routing weights [T,K]."""
    rng = _np_rng(seed, 1)
    if T == 0:
        return np.zeros((0, K), np.int32), np.zeros((0, K), np.float32)
    if kind[0] == "uniform":
        ids = np.argsort(rng.random((T, E_total)), axis=1)[:, :K]
    elif kind[0] == "zipf":
        s = float(kind[1])
        rank_of = rng.permutation(E_total)              # rank of expert e
        logp = -s * np.log(rank_of + 1.0)
        gumbel = -np.log(-np.log(rng.random((T, E_total))))
        ids = np.argsort(-(logp[None, :] + gumbel), axis=1)[:, :K]
    else:
        raise ValueError(kind)
    logits = _np_rng(seed, 2).standard_normal((T, K))
    w = np.exp(logits - logits.max(1, keepdims=True))
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    return ids.astype(np.int32), w


# --------------------------------------------------------------------------
# storage-format packing (data preparation)
# --------------------------------------------------------------------------

def _e2m1_codes(y: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code of each |y| <= 6 (ties to the even code), sign in bit 3."""
    grid = torch.tensor(_E2M1_GRID, dtype=y.dtype, device=y.device)
    a = y.abs().clamp(max=6.0)
    lo = (torch.bucketize(a, grid, right=True) - 1).clamp(0, 7)
    hi = (lo + 1).clamp(max=7)
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    take_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0) & (hi != lo))
    code = torch.where(take_hi, hi, lo)
    return (code | (torch.signbit(y).to(code.dtype) << 3)).to(torch.uint8)


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """[..., n] codes -> [..., n/2] bytes, element 2i in the low nibble."""
    c = codes.reshape(*codes.shape[:-1], codes.shape[-1] // 2, 2)
    return (c[..., 0] | (c[..., 1] << 4)).contiguous()


def pack_mxfp4(x: torch.Tensor):
    """fp32 [..., n] -> (packed uint8 [..., n/2], UE8M0 uint8 [..., n/32])."""
    shp = x.shape
    b = x.reshape(-1, 32).float()
    amax = b.abs().amax(1)
    m, p = torch.frexp(amax)                       # amax = m * 2^p, m in [0.5, 1)
    e = torch.where(m * 8.0 <= 6.0, p - 3, p - 2)  # smallest e with amax*2^-e <= 6
    e = torch.where(amax > 0, e, torch.full_like(e, -127)).clamp(-127, 127)
    y = torch.ldexp(b, (-e).float()[:, None])
    codes = _e2m1_codes(y).reshape(shp)
    return _pack_nibbles(codes), (e + 127).to(torch.uint8).reshape(*shp[:-1], shp[-1] // 32)


def pack_nvfp4(x: torch.Tensor, gscale: torch.Tensor):
    """fp32 [..., n] with an fp32 global scale per leading index (broadcast
    over the trailing dims) -> (packed uint8 [..., n/2], E4M3 uint8 [..., n/16])."""
    shp = x.shape
    b = x.float().reshape(*shp[:-1], shp[-1] // 16, 16)
    g = gscale.float().reshape(*gscale.shape, *([1] * (b.dim() - gscale.dim())))
    amax = b.abs().amax(-1, keepdim=True)
    s8 = (amax / (6.0 * g)).to(torch.float8_e4m3fn)
    denom = s8.float() * g
    y = torch.where(denom > 0, b / torch.where(denom > 0, denom, torch.ones_like(denom)),
                    torch.zeros_like(b))
    codes = _e2m1_codes(y).reshape(shp)
    return _pack_nibbles(codes), s8.squeeze(-1).view(torch.uint8).contiguous()


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    T: int
    H: int
    I: int
    E_total: int
    E_loc: int
    off: int
    K: int
    act: int
    wt: int
    device: str
    topk_ids: torch.Tensor          # int32 [T,K] (device)
    topk_weights: torch.Tensor      # fp32 [T,K]
    x_bf16: torch.Tensor            # bf16 [T,H]
    w1: torch.Tensor                # uint8 [E_loc, 2I, H/2]
    w1_scale: torch.Tensor          # uint8 [E_loc, 2I, H/32 or H/16]
    w2: torch.Tensor                # uint8 [E_loc, H, I/2]
    w2_scale: torch.Tensor          # uint8 [E_loc, H, I/32 or I/16]
    gemm1_alpha: torch.Tensor       # fp32 [E_loc]
    gemm1_beta: torch.Tensor        # fp32 [E_loc]
    g1_alphas: Optional[torch.Tensor] = None
    g1_alphas_up: Optional[torch.Tensor] = None
    g2_alphas: Optional[torch.Tensor] = None
    w1_gscale: Optional[torch.Tensor] = None   # fp32 [E_loc, 2] (NVFP4)
    w2_gscale: Optional[torch.Tensor] = None   # fp32 [E_loc]    (NVFP4)
    x_q: Optional[torch.Tensor] = None         # NVFP4 packed activations [T, H/2]
    x_scale: Optional[torch.Tensor] = None     # NVFP4 E4M3 [T, H/16]
    x_gscale: Optional[torch.Tensor] = None    # NVFP4 fp32 [T]

    def host(self, name: str) -> Optional[np.ndarray]:
        """numpy copy of a field (bf16 tensors come back as uint16 bits)."""
        t = getattr(self, name)
        if t is None:
            return None
        t = t.detach()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).cpu().numpy().view(np.uint16)
        return t.cpu().numpy()


def make(name: str = "tiny", *, device="cpu", seed: int = 0, T: Optional[int] = None,
         beta: Optional[float] = None, beta_lin: Optional[float] = None, **overrides) -> Workload:
    """Build a seeded workload.  ``T``, ``beta``/``beta_lin`` (constant SiTU
    caps, e.g. Kimi-K3's 4.0 / 25.0) and any CONFIGS field may be overridden."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    if T is not None:
        cfg["T"] = T
    T, H, I, E, E_loc, off, K = (cfg[k] for k in ("T", "H", "I", "E_total", "E_loc", "off", "K"))
    act, wt = cfg["act"], cfg["wt"]
    dev = torch.device(device)

    ids, wts = routing(T, K, E, cfg["routing"], seed)
    x = torch.from_numpy(_np_rng(seed, 3).standard_normal((T, H), dtype=np.float32))
    x_bf16 = x.to(torch.bfloat16).to(dev)

    bs = 16 if wt == W_NVFP4 else 32
    w1 = torch.empty((E_loc, 2 * I, H // 2), dtype=torch.uint8, device=dev)
    w1s = torch.empty((E_loc, 2 * I, H // bs), dtype=torch.uint8, device=dev)
    w2 = torch.empty((E_loc, H, I // 2), dtype=torch.uint8, device=dev)
    w2s = torch.empty((E_loc, H, I // bs), dtype=torch.uint8, device=dev)
    w1g = torch.empty((E_loc, 2), dtype=torch.float32, device=dev) if wt == W_NVFP4 else None
    w2g = torch.empty((E_loc,), dtype=torch.float32, device=dev) if wt == W_NVFP4 else None
    chunk = 16
    for c0 in range(0, E_loc, chunk):
        c1 = min(E_loc, c0 + chunk)
        gen = _torch_gen(seed, 100 + c0 // chunk, dev)
        a1 = torch.randn((c1 - c0, 2 * I, H), generator=gen, device=dev) * 0.02
        a2 = torch.randn((c1 - c0, H, I), generator=gen, device=dev) * 0.02
        if wt == W_MXFP4:
            w1[c0:c1], w1s[c0:c1] = pack_mxfp4(a1)
            w2[c0:c1], w2s[c0:c1] = pack_mxfp4(a2)
        else:
            halves = a1.reshape(c1 - c0, 2, I, H)
            g1 = halves.abs().amax(dim=(2, 3)) / (6.0 * 448.0)          # [n, 2]
            p1, s1 = pack_nvfp4(halves, g1)
            w1[c0:c1] = p1.reshape(c1 - c0, 2 * I, H // 2)
            w1s[c0:c1] = s1.reshape(c1 - c0, 2 * I, H // 16)
            w1g[c0:c1] = g1
            g2 = a2.abs().amax(dim=(1, 2)) / (6.0 * 448.0)
            w2[c0:c1], w2s[c0:c1] = pack_nvfp4(a2, g2)
            w2g[c0:c1] = g2
        del a1, a2

    prng = _np_rng(seed, 4)
    if cfg["params"] == "unit":
        b = np.ones(E_loc, np.float32)
        bl = np.zeros(E_loc, np.float32)
        ag = np.ones(E_loc, np.float32)
        au = np.ones(E_loc, np.float32)
    else:
        b = prng.uniform(0.5, 1.5, E_loc).astype(np.float32)
        bl = prng.uniform(0.0, 0.1, E_loc).astype(np.float32)
        ag = prng.uniform(0.9, 1.1, E_loc).astype(np.float32)
        au = prng.uniform(0.9, 1.1, E_loc).astype(np.float32)
    if beta is not None:
        b = np.full(E_loc, beta, np.float32)
    if beta_lin is not None:
        bl = np.full(E_loc, beta_lin, np.float32)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    wl = Workload(name=name, T=T, H=H, I=I, E_total=E, E_loc=E_loc, off=off, K=K, act=act, wt=wt,
                  device=str(dev), topk_ids=t(ids), topk_weights=t(wts), x_bf16=x_bf16,
                  w1=w1, w1_scale=w1s, w2=w2, w2_scale=w2s, gemm1_alpha=t(b), gemm1_beta=t(bl),
                  g1_alphas=t(ag), g1_alphas_up=t(au), g2_alphas=None,
                  w1_gscale=w1g, w2_gscale=w2g)
    if act == ACT_NVFP4:
        xf = x_bf16.float()
        gs = xf.abs().amax(1) / (6.0 * 448.0) if T > 0 else torch.zeros(0, device=dev)
        gs = torch.where(gs > 0, gs, torch.ones_like(gs))
        wl.x_q, wl.x_scale = pack_nvfp4(xf, gs)
        wl.x_gscale = gs.float().contiguous()
    return wl


def oracle_kwargs(wl: Workload, *, x_q=None, x_scale=None, x_gscale=None) -> dict:
    """Host (numpy) keyword arguments for the oracle's ``moe_forward``.  For
    the MXFP8 chain pass the oracle's own quantised activations; for NVFP4
    they may be passed too (default: this module's host packing)."""
    kw = dict(T=wl.T, H=wl.H, I=wl.I, num_experts_total=wl.E_total,
              num_local_experts=wl.E_loc, local_expert_offset=wl.off, top_k=wl.K,
              act=wl.act, wt=wl.wt, topk_ids=wl.host("topk_ids"),
              topk_weights=wl.host("topk_weights"), w1=wl.host("w1"),
              w1_scale=wl.host("w1_scale"), w2=wl.host("w2"), w2_scale=wl.host("w2_scale"),
              gemm1_alpha=wl.host("gemm1_alpha"), gemm1_beta=wl.host("gemm1_beta"),
              g1_alphas=wl.host("g1_alphas"), g1_alphas_up=wl.host("g1_alphas_up"),
              g2_alphas=wl.host("g2_alphas"), w1_gscale=wl.host("w1_gscale"),
              w2_gscale=wl.host("w2_gscale"))
    if wl.act == ACT_BF16:
        kw["hidden_states"] = wl.host("x_bf16")
    elif wl.act == ACT_MXFP8:
        kw["hidden_states_q"], kw["hidden_states_scale"] = x_q, x_scale
    else:
        kw["hidden_states_q"] = wl.host("x_q") if x_q is None else x_q
        kw["hidden_states_scale"] = wl.host("x_scale") if x_scale is None else x_scale
        kw["hidden_states_gscale"] = wl.host("x_gscale") if x_gscale is None else x_gscale
    return kw
