"""Pins for the oracle's permute, SiTU and routed-MoE forward.

The oracle is checked against things other than itself:
  * SiTU: its beta -> infinity limit (SwiGLU, the golden `_swiglu_act` of
    TensorRT-LLM PR #17865), the tanh-free identity that PR's "SiTU in the
    kernel" commit validated at Kimi-K3's beta=4 / linear beta=25, and its
    symmetries;
  * permute: numpy's stable argsort, and the bijection / count invariants;
  * forward: a token-major brute-force loop (the golden per-token, per-slot
    reference MoE of the same PR) that dequantises through the hand-written
    E2M1 table and torch's float8 decoders; a dense special case against
    numpy matmul; the invariants of routing (zero weight, filtered tokens,
    linearity in routing weights) and of sharding (8 partial outputs sum to
    the unsharded one).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden
from block_scaled_fp4_permute_gb300 import workloads as W

E2M1 = np.array([float(v) for _, v in golden("e2m1_values.txt")])
K3 = {r[0]: float(r[1]) for r in golden("situ_k3.txt")}


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


# --------------------------------------------------------------------------
# SiTU
# --------------------------------------------------------------------------

def test_situ_large_caps_reduce_to_swiglu():
    rng = np.random.default_rng(0)
    for g, u in rng.standard_normal((200, 2)) * 3:
        ref = g * sigmoid(g) * u
        assert oracle.situ(g, u, 1e7, 1e7) == pytest.approx(ref, rel=1e-6, abs=1e-12)


def test_situ_nonpositive_cap_is_the_limit():
    for g, u in [(0.3, -1.2), (-2.0, 4.0), (5.0, 0.5)]:
        assert oracle.situ(g, u, 0.0, 0.0) == pytest.approx(g * sigmoid(g) * u, rel=1e-15)
        assert oracle.situ(g, u, -1.0, 2.0) == pytest.approx(
            g * sigmoid(g) * 2.0 * math.tanh(u / 2.0), rel=1e-15)


def test_situ_tanh_free_identity_at_k3_constants():
    beta, beta_lin, tol = K3["beta"], K3["linear_beta"], K3["max_rel_err"]
    rng = np.random.default_rng(1)
    worst = 0.0
    for g, u in rng.standard_normal((2000, 2)) * 8:
        ident = (2 * beta * sigmoid(2 * g / beta) - beta) * sigmoid(g) * \
                (2 * beta_lin * sigmoid(2 * u / beta_lin) - beta_lin)
        got = oracle.situ(g, u, beta, beta_lin)
        worst = max(worst, abs(got - ident) / max(abs(ident), 1e-300))
    assert worst <= tol


def test_situ_symmetries_and_saturation():
    b, bl = 1.3, 0.07
    for g, u in [(0.4, 0.9), (-1.1, 2.5), (3.0, -0.2)]:
        assert oracle.situ(g, -u, b, bl) == -oracle.situ(g, u, b, bl)       # odd in u
    assert oracle.situ(0.0, 3.0, b, bl) == 0.0
    assert oracle.situ(2.0, 0.0, b, bl) == 0.0
    # both factors saturate at their caps: gate -> beta, up -> beta_lin
    assert oracle.situ(200.0, 200.0, b, bl) == pytest.approx(b * bl, rel=1e-12)
    # gate vanishes for very negative g (sigmoid -> 0)
    assert abs(oracle.situ(-60.0, 1.0, b, bl)) < 1e-20


# --------------------------------------------------------------------------
# permute
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,K,E_total,E_loc,off", [(16, 2, 8, 8, 0), (37, 5, 20, 6, 7),
                                                   (100, 16, 896, 112, 336), (1, 3, 4, 4, 0),
                                                   (0, 4, 8, 8, 0)])
def test_permute_matches_stable_sort(T, K, E_total, E_loc, off):
    rng = np.random.default_rng(T * 7 + K)
    ids = rng.integers(-2, E_total + 2, (T, K)).astype(np.int32)   # incl. out-of-range IDs
    counts, offsets, psrc, s2r, R = oracle.permute(ids, E_total, E_loc, off)
    flat = ids.reshape(-1)
    kept = (flat >= off) & (flat < off + E_loc)
    slots = np.nonzero(kept)[0]
    order = slots[np.argsort(flat[slots] - off, kind="stable")]
    assert R == kept.sum() == counts.sum() == offsets[-1]
    assert np.array_equal(psrc[:R], order)
    assert np.all(psrc[R:] == -1)
    assert np.array_equal(counts, np.bincount(flat[slots] - off, minlength=E_loc))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    # bijection between kept slots and rows
    assert np.all(s2r[~kept] == -1)
    assert np.array_equal(np.sort(s2r[kept]), np.arange(R))
    assert np.array_equal(psrc[s2r[kept]], slots)


# --------------------------------------------------------------------------
# brute-force forward (token-major, per slot)
# --------------------------------------------------------------------------

def _dq_fp4(packed, scales, nvfp4):
    codes = np.stack([packed & 15, packed >> 4], -1).reshape(*packed.shape[:-1], -1)
    dt = torch.float8_e4m3fn if nvfp4 else torch.float8_e8m0fnu
    sc = torch.from_numpy(np.ascontiguousarray(scales)).view(dt).double().numpy()
    return E2M1[codes] * np.repeat(sc, 16 if nvfp4 else 32, axis=-1)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def _mxfp8_round_trip(h32):
    """Per-32 MXFP8 round trip of fp32 values: scale from the fp32 bits in
    closed form (amax = m*2^k, e = k-8+(m>1.75)), elements by torch."""
    out = np.empty(h32.shape, np.float64)
    for b in range(0, h32.shape[0], 32):
        blk = h32[b:b + 32].astype(np.float32)
        amax = np.float32(np.abs(blk).max())
        if amax == 0:
            e = -127
        else:
            bits = int(amax.view(np.uint32))
            k = ((bits >> 23) & 0xFF) - 127
            e = max(-127, k - 8 + (1 if (bits & 0x7FFFFF) > 0x600000 else 0))
        q = torch.from_numpy((blk.astype(np.float64) * 2.0 ** -e).astype(np.float32)).to(
            torch.float8_e4m3fn).double().numpy()
        out[b:b + 32] = q * 2.0 ** e
    return out


def _situ_np(g, u, beta, beta_lin):
    gate = beta * np.tanh(g / beta) * sigmoid(g) if beta > 0 else g * sigmoid(g)
    up = beta_lin * np.tanh(u / beta_lin) if beta_lin > 0 else u
    return gate * up


def _swiglu_bias_np(g, u, alpha, beta):
    return g * sigmoid(g * alpha) * (u + beta)


def _nvfp4_round_trip(h_bf16_values):
    """H1 (bf16 values, one row) requantised per token to NVFP4 with the
    oracle's own quantiser (pinned in test_oracle_formats against an
    independent torch formulation), dequantised exactly here."""
    bits = torch.from_numpy(np.ascontiguousarray(h_bf16_values, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)[None, :]
    q, s, g = oracle.quant_nvfp4(bits)
    return _dq_fp4(q, s, True)[0] * float(g[0])


def brute_force(kw, alpha_power=1, activation=0, topk_in_fc1=0, h1_nvfp4=0):
    T, H, I, K = kw["T"], kw["H"], kw["I"], kw["top_k"]
    off, E_loc = kw["local_expert_offset"], kw["num_local_experts"]
    act, nv = kw["act"], kw["wt"] == W.W_NVFP4
    ones = np.ones(E_loc)
    ag = kw["g1_alphas"] if kw["g1_alphas"] is not None else ones
    au = kw["g1_alphas_up"] if kw["g1_alphas_up"] is not None else ones
    a2 = kw["g2_alphas"] if kw["g2_alphas"] is not None else ones
    if act == W.ACT_BF16:
        X = torch.from_numpy(kw["hidden_states"].view(np.int16)).view(torch.bfloat16).double().numpy()
        xg = np.ones(T)
    elif act == W.ACT_MXFP8:
        X = torch.from_numpy(kw["hidden_states_q"]).view(torch.float8_e4m3fn).double().numpy() * \
            np.repeat(torch.from_numpy(kw["hidden_states_scale"]).view(torch.float8_e8m0fnu)
                      .double().numpy(), 32, axis=1)
        xg = np.ones(T)
    else:
        X = _dq_fp4(kw["hidden_states_q"], kw["hidden_states_scale"], True)
        xg = kw["hidden_states_gscale"].astype(np.float64)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(K):
            e = int(kw["topk_ids"][t, j]) - off
            if not 0 <= e < E_loc:
                continue
            W1 = _dq_fp4(kw["w1"][e], kw["w1_scale"][e], nv)
            W2 = _dq_fp4(kw["w2"][e], kw["w2_scale"][e], nv)
            g1g, g1u = (kw["w1_gscale"][e] if nv else (1.0, 1.0))
            g2 = kw["w2_gscale"][e] if nv else 1.0
            g = ag[e] ** alpha_power * g1g * xg[t] * (W1[:I] @ X[t])
            u = au[e] ** alpha_power * g1u * xg[t] * (W1[I:] @ X[t])
            fn = _swiglu_bias_np if activation == oracle.ACT_FN_SWIGLU_BIAS else _situ_np
            a = fn(g, u, kw["gemm1_alpha"][e], kw["gemm1_beta"][e])
            w = float(kw["topk_weights"][t, j])
            if topk_in_fc1:
                a = a * w                  # the routing weight scales H1 before its rounding
            a = a.astype(np.float32)
            h = _mxfp8_round_trip(a) if act == W.ACT_MXFP8 else _bf16(a)
            if nv and h1_nvfp4:
                h = _nvfp4_round_trip(h)
            y = a2[e] * g2 * (W2 @ h)
            out[t] += (1.0 if topk_in_fc1 else w) * y
    return out


def _small(act=W.ACT_BF16, wt=W.W_MXFP4, seed=0, **kw):
    base = dict(T=9, H=64, I=32, E_total=12, E_loc=5, off=4, K=3, params="k3_random",
                act=act, wt=wt)
    base.update(kw)
    return W.make("tiny", seed=seed, **base)


def _kwargs(wl):
    if wl.act == W.ACT_MXFP8:
        q, s = oracle.quant_mxfp8(wl.host("x_bf16"))
        return W.oracle_kwargs(wl, x_q=q, x_scale=s)
    return W.oracle_kwargs(wl)


def _close(a, b, rel=1e-9):
    scale = max(np.sqrt(np.mean(b ** 2)), 1e-300)
    assert np.max(np.abs(a - b)) <= rel * scale, np.max(np.abs(a - b)) / scale


def test_tiny_config_matches_brute_force():
    wl = W.make("tiny")
    kw = _kwargs(wl)
    _close(oracle.moe_forward(**kw), brute_force(kw))


@pytest.mark.parametrize("act,wt", [(W.ACT_BF16, W.W_MXFP4), (W.ACT_MXFP8, W.W_MXFP4),
                                    (W.ACT_NVFP4, W.W_NVFP4)])
@pytest.mark.parametrize("seed", [1, 2])
def test_small_shards_match_brute_force(act, wt, seed):
    wl = _small(act, wt, seed)
    kw = _kwargs(wl)
    ids = kw["topk_ids"].copy()
    ids[0, 1] = ids[0, 0]               # a duplicate ID contributes twice
    ids[1, :] = 0                        # a token routed only outside the shard
    ids[2, 2] = -1                       # a negative ID is dropped
    kw["topk_ids"] = ids
    got = oracle.moe_forward(**kw)
    ref = brute_force(kw)
    _close(got, ref, rel=1e-7)           # MXFP8 rounding decisions match exactly
    assert np.all(got[1] == 0.0)
    assert np.sqrt(np.mean(ref ** 2)) > 0


def test_token_subset_equals_rows_of_full_output():
    wl = _small(seed=3, T=20)
    kw = _kwargs(wl)
    full = oracle.moe_forward(**kw)
    toks = np.array([19, 0, 7, 7, 3], np.int32)
    assert np.array_equal(oracle.moe_forward(**kw, tokens=toks), full[toks])


def test_dense_special_case_matches_matmul():
    # one expert, top-1, routing weight 1, caps off (SwiGLU), unit alphas:
    # the layer is the dense MLP  bf16(SwiGLU(X W_gate^T, X W_up^T)) W2^T
    wl = W.make("tiny", T=24, H=96, I=64, E_total=1, E_loc=1, off=0, K=1, beta=0.0,
                beta_lin=0.0)
    kw = _kwargs(wl)
    kw["topk_weights"] = np.ones_like(kw["topk_weights"])
    X = torch.from_numpy(kw["hidden_states"].view(np.int16)).view(torch.bfloat16).double().numpy()
    W1 = _dq_fp4(kw["w1"][0], kw["w1_scale"][0], False)
    W2 = _dq_fp4(kw["w2"][0], kw["w2_scale"][0], False)
    G, U = X @ W1[:64].T, X @ W1[64:].T
    Hh = _bf16((G * sigmoid(G) * U).astype(np.float32))
    _close(oracle.moe_forward(**kw), Hh @ W2.T)


def test_zero_routing_weight_contributes_nothing():
    wl = _small(seed=4)
    kw = _kwargs(wl)
    w = kw["topk_weights"].copy()
    w[3, 1] = 0.0
    kw["topk_weights"] = w
    base = oracle.moe_forward(**kw)
    ids = kw["topk_ids"].copy()
    ids[3, 1] = 4 + (ids[3, 1] - 4 + 1) % 5        # another local expert
    kw["topk_ids"] = ids
    assert np.array_equal(oracle.moe_forward(**kw), base)


def test_linear_in_routing_weights():
    wl = _small(seed=5)
    kw = _kwargs(wl)
    base = oracle.moe_forward(**kw)
    kw["topk_weights"] = kw["topk_weights"] * 2.0
    _close(oracle.moe_forward(**kw), 2.0 * base, rel=1e-14)


def test_eight_shard_partials_sum_to_unsharded():
    wl = _small(seed=6, T=11, E_total=16, E_loc=16, off=0, K=4)
    kw = _kwargs(wl)
    full = oracle.moe_forward(**kw)
    acc = np.zeros_like(full)
    for r in range(8):
        sk = dict(kw)
        sl = slice(2 * r, 2 * r + 2)
        sk.update(num_local_experts=2, local_expert_offset=2 * r)
        for k in ("w1", "w1_scale", "w2", "w2_scale", "gemm1_alpha", "gemm1_beta", "g1_alphas",
                  "g1_alphas_up"):
            sk[k] = kw[k][sl]
        acc += oracle.moe_forward(**sk)
    _close(acc, full, rel=1e-12)


def test_double_applied_alpha_is_detected():
    """A planted mistake: applying g1_alphas / g1_alphas_up twice (the kind of
    repeated scale application the PR's strict xfail records) must move the
    output well outside the parity tolerance."""
    wl = _small(seed=7, beta=4.0, beta_lin=25.0)
    kw = _kwargs(wl)
    kw["g1_alphas"] = np.full(5, 1.5, np.float32)
    kw["g1_alphas_up"] = np.full(5, 0.6, np.float32)
    good = oracle.moe_forward(**kw)
    _close(good, brute_force(kw), rel=1e-9)
    bad = brute_force(kw, alpha_power=2)
    rms = np.sqrt(np.mean(good ** 2))
    assert np.max(np.abs(bad - good)) > 0.2 * rms


# --------------------------------------------------------------------------
# activation variants: SwigluBias, apply_topk_in_fc1
# --------------------------------------------------------------------------

def test_swiglu_bias_at_unit_alpha_zero_beta_is_swiglu():
    """SwigluBias(alpha=1, beta=0) and SiTU with both caps off are both SwiGLU
    g * sigmoid(g) * u, written as two different oracle functions."""
    rng = np.random.default_rng(21)
    for g, u in rng.normal(0, 4, (200, 2)):
        assert oracle.swiglu_bias(g, u, 1.0, 0.0) == pytest.approx(oracle.situ(g, u, 0.0, 0.0), rel=1e-14, abs=1e-300)


def test_swiglu_bias_shift_and_gate_limits():
    rng = np.random.default_rng(22)
    for g, u, a, b in rng.normal(0, 2, (200, 4)):
        a = abs(a) + 0.1
        # beta shifts the linear input
        assert oracle.swiglu_bias(g, u, a, b) == pytest.approx(oracle.swiglu_bias(g, u + b, a, 0.0), rel=1e-12)
    # a steep gate: sigmoid(alpha g) -> step(g)
    assert oracle.swiglu_bias(2.0, 3.0, 1e4, 0.5) == pytest.approx(2.0 * 3.5, rel=1e-12)
    assert abs(oracle.swiglu_bias(-2.0, 3.0, 1e4, 0.5)) < 1e-300


@pytest.mark.parametrize("act,wt", [(W.ACT_BF16, W.W_MXFP4), (W.ACT_MXFP8, W.W_MXFP4),
                                    (W.ACT_NVFP4, W.W_NVFP4)])
@pytest.mark.parametrize("activation,topk_in_fc1", [(1, 0), (0, 1), (1, 1)])
def test_variants_match_brute_force(act, wt, activation, topk_in_fc1):
    wl = _small(act, wt, 3)
    kw = _kwargs(wl)
    if activation == 1:   # SwigluBias alpha ~ 1.7, beta ~ small
        kw["gemm1_alpha"] = np.full_like(kw["gemm1_alpha"], 1.702)
        kw["gemm1_beta"] = np.linspace(-0.5, 0.5, kw["gemm1_beta"].shape[0]).astype(np.float32)
    got = oracle.moe_forward(**kw, activation=activation, apply_topk_in_fc1=topk_in_fc1)
    ref = brute_force(kw, activation=activation, topk_in_fc1=topk_in_fc1)
    _close(got, ref, rel=1e-7)
    assert np.sqrt(np.mean(ref ** 2)) > 0


def test_topk_in_fc1_differs_only_by_rounding_position():
    """FC2 is linear, so moving the routing weight from the FC2 output to H1
    changes only where H1 is rounded to bf16: the two outputs differ by
    rounding-sized amounts, well inside the layer's parity bar (2% of rms),
    and are not identical."""
    wl = _small(W.ACT_BF16, W.W_MXFP4, 4)
    kw = _kwargs(wl)
    a = oracle.moe_forward(**kw)
    b = oracle.moe_forward(**kw, apply_topk_in_fc1=1)
    rms = np.sqrt(np.mean(a ** 2))
    assert np.max(np.abs(a - b)) <= 2e-2 * rms
    assert np.sqrt(np.mean((a - b) ** 2)) <= 2.0 ** -8 * rms
    assert not np.array_equal(a, b)


# ---------------------------------------------------------------------------
# NVFP4 chain with H1 requantised per token (FlashInfer 0.6.18 MoE-LoRA AOT
# release notes, "Summary": per-token NVFP4 activation scaling; the prior art
# quantises the activation unfused)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [1, 2, 3])
def test_h1_nvfp4_matches_brute_force(seed):
    wl = _small(W.ACT_NVFP4, W.W_NVFP4, seed, I=64)
    kw = _kwargs(wl)
    _close(oracle.moe_forward(**kw, h1_nvfp4=1), brute_force(kw, h1_nvfp4=1))


def test_h1_nvfp4_is_the_bf16_chain_within_the_nvfp4_error():
    """Requantising H1 moves each FC2 input by at most half an E2M1 step of
    its block (the quantiser's rounding), so the output stays within the
    bound that error implies, and it does move (the option is not a no-op)."""
    wl = _small(W.ACT_NVFP4, W.W_NVFP4, 4, T=16, I=64, H=128)
    kw = _kwargs(wl)
    ref = oracle.moe_forward(**kw)
    got = oracle.moe_forward(**kw, h1_nvfp4=1)
    assert not np.array_equal(ref, got)
    rel = np.sqrt(np.mean((got - ref) ** 2)) / np.sqrt(np.mean(ref ** 2))
    # E2M1 has one mantissa bit: relative rounding error up to 1/3 per
    # element at the block maximum's binade, smaller on average
    assert 1e-3 < rel < 0.25, rel


def test_h1_nvfp4_on_an_exactly_representable_h1_is_the_bf16_chain():
    """When every H1 value is an E2M1 code times a power of two that the
    quantiser reproduces, requantising changes nothing: with SwiGLU (both
    caps off), unit alphas and a W1 whose up half is zero except one row,
    H1 has one non-zero element per row, which NVFP4 holds exactly (it is
    its block's and row's maximum: code 6 under the scale 448 * gs)."""
    wl = _small(W.ACT_NVFP4, W.W_NVFP4, 5, T=6, I=32, H=64, K=1, E_total=4, E_loc=4, off=0)
    kw = _kwargs(wl)
    kw["gemm1_alpha"] = np.zeros_like(kw["gemm1_alpha"])
    kw["gemm1_beta"] = np.zeros_like(kw["gemm1_beta"])
    w1 = kw["w1"].copy()
    w1[:, 32 + 1:, :] = 0            # up rows other than row 0 give u = 0
    kw["w1"] = w1
    ref = oracle.moe_forward(**kw)
    got = oracle.moe_forward(**kw, h1_nvfp4=1)
    # one non-zero h per row: its NVFP4 round trip is the bf16 value times
    # (6 * E4M3(448) * gs) / (amax) = 1 up to the fp32 steps of the rule
    _close(got, ref, rel=1e-6)
