"""Pins for the oracle's number formats and MXFP8 quantisation.

Each check compares the oracle with something other than itself: hand-written
tables (tests/golden), torch's own float8 decoders/encoders (library
routines), closed forms and defining properties.
"""
import math

import numpy as np
import torch

import oracle
from conftest import golden


def test_e2m1_table_by_hand():
    rows = golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        v = oracle.e2m1_value(int(code))
        assert v == float(val)
        assert math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e4m3_hand_values():
    for code, val in golden("e4m3_values.txt"):
        v = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))


def test_e4m3_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_ue8m0_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([oracle.ue8m0_value(c) for c in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])


def test_bf16_round_trip_matches_torch():
    rng = np.random.default_rng(1)
    f = np.concatenate([rng.standard_normal(2000), rng.standard_normal(200) * 1e-30,
                        rng.standard_normal(200) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(x)) for x in f], np.uint16)
    assert np.array_equal(ref, got)
    back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(back, np.array([oracle.bf16_value(int(h)) for h in ref]))


def test_e4m3_encode_matches_torch_including_ties():
    vals = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (vals[1:] + vals[:-1]) / 2            # exact ties between neighbours
    rng = np.random.default_rng(2)
    rnd = rng.uniform(-448, 448, 5000)
    tiny = rng.uniform(-0.02, 0.02, 2000)
    xs = np.concatenate([vals, -vals, mids, -mids, rnd, tiny]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates():
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-500.0) == 0xFE


def _closed_form_exponent(bf16_bits):
    """ceil(log2(amax/448)) from the bf16 bits: amax = m * 2^k, m in [1, 2),
    448 = 1.75 * 2^8, so e = k - 8 + (m > 1.75).  Normal bf16 only."""
    k = ((bf16_bits >> 7) & 0xFF) - 127
    mant = bf16_bits & 0x7F
    return k - 8 + (1 if mant > 0x60 else 0)      # 1.75 = 1 + 0x60/128


def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_mxfp8_exponent_closed_form_and_minimality():
    rng = np.random.default_rng(3)
    f = np.abs(rng.standard_normal(4000) * np.exp2(rng.integers(-60, 60, 4000))).astype(np.float32)
    for h in _bf16_bits(f):
        amax = oracle.bf16_value(int(h))
        e = oracle.mxfp8_exponent(amax)
        assert e == _closed_form_exponent(int(h))
        assert amax * 2.0 ** -e <= 448.0 < amax * 2.0 ** -(e - 1)
    # boundaries: exactly 448 * 2^j needs e = j; just above needs j + 1
    for j in (-5, 0, 3):
        assert oracle.mxfp8_exponent(448.0 * 2.0 ** j) == j
        assert oracle.mxfp8_exponent(np.nextafter(448.0, 1e9) * 2.0 ** j) == j + 1
    assert oracle.mxfp8_exponent(0.0) == -127
    assert oracle.mxfp8_exponent(1e-45) == -127


def test_quant_mxfp8_matches_library_rounding():
    rng = np.random.default_rng(4)
    T, H = 7, 256
    x = rng.standard_normal((T, H)).astype(np.float32)
    x[0, :32] = 0.0                       # an all-zero block
    x[1, 32:64] *= 1e-3                   # a small-magnitude block
    x[2, 64:96] = -0.0                    # negative zeros
    x[3, 96:128] *= 1e4
    bits = _bf16_bits(x)
    q, s = oracle.quant_mxfp8(bits)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for t in range(T):
        for b in range(H // 32):
            blk = xb[t, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            e = -127 if amax == 0 else _closed_form_exponent(int(_bf16_bits([amax])[0]))
            assert s[t, b] == e + 127
            ref = torch.from_numpy((blk * 2.0 ** -e).astype(np.float32)).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[t, 32 * b:32 * b + 32], ref)
    assert np.all(q[0, :32] == 0) and s[0, 0] == 0
    assert np.all(q[2, 64:96] == 0x80)


def test_quant_mxfp8_round_trip_error_bound():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 512)).astype(np.float32)
    bits = _bf16_bits(x)
    q, s = oracle.quant_mxfp8(bits)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    sc = np.repeat(torch.from_numpy(s).view(torch.float8_e8m0fnu).double().numpy(), 32, axis=1)
    dq = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy() * sc
    # a normal E4M3 element is within 2^-4 relative; a subnormal within half
    # its step of 2^-9 (times the block scale)
    assert np.all(np.abs(dq - xb) <= np.maximum(np.abs(xb) * 2.0 ** -4, sc * 2.0 ** -10))
    # values already on the grid survive exactly (the codes may change: when
    # amax rounds down to 224 * 2^e the next pass picks the scale 2^(e-1))
    q2, s2 = oracle.quant_mxfp8(_bf16_bits(dq))
    sc2 = np.repeat(torch.from_numpy(s2).view(torch.float8_e8m0fnu).double().numpy(), 32, axis=1)
    assert np.array_equal(torch.from_numpy(q2).view(torch.float8_e4m3fn).double().numpy() * sc2, dq)


# ---------------------------------------------------------------------------
# NVFP4 activation quantisation (per-token global scale, E4M3 per 16, E2M1)
# ---------------------------------------------------------------------------

def _e2m1_brute(v):
    """Nearest of the 16 signed E2M1 values by exhaustive comparison, ties to
    the even code, saturating; a negative value rounding to 0 keeps the sign."""
    vals = [oracle.e2m1_value(c) for c in range(8)]
    a = min(abs(v), 6.0)
    best = min(range(8), key=lambda c: (abs(a - vals[c]), c % 2))
    return best | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_encode_brute_force_and_ties():
    rng = np.random.default_rng(11)
    pts = list(rng.uniform(-7.5, 7.5, 4000))
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [(grid[i] + grid[i + 1]) / 2 for i in range(7)]     # every tie
    for m in mids:
        pts += [m, -m, np.nextafter(m, 0.0), np.nextafter(m, 10.0)]
    pts += [0.0, -0.0, 6.0, 1e9, -1e9]
    for v in pts:
        assert oracle.e2m1_encode(v) == _e2m1_brute(float(v)), v


def _bits(x):
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quant_nvfp4_matches_torch_packing():
    """Against an independent torch formulation of the same fp32 steps
    (float8_e4m3fn casts and a bucketed E2M1 search): identical bytes."""
    from block_scaled_fp4_permute_gb300 import workloads as W
    g = torch.Generator().manual_seed(5)
    x = torch.randn((48, 512), generator=g) * torch.logspace(-3, 3, 48).unsqueeze(1)
    x[3, :] = 0.0
    x[4, 17] = -0.0
    xb = x.to(torch.bfloat16)
    q, s, gs = oracle.quant_nvfp4(_bits(xb))
    xf = xb.float()
    ref_gs = xf.abs().amax(1) / (6.0 * 448.0)
    ref_gs = torch.where(ref_gs > 0, ref_gs, torch.ones_like(ref_gs))
    rq, rs = W.pack_nvfp4(xf, ref_gs)
    assert np.array_equal(gs, ref_gs.numpy())
    assert np.array_equal(s, rs.numpy())
    assert np.array_equal(q, rq.numpy())


def test_quant_nvfp4_properties():
    g = torch.Generator().manual_seed(6)
    x = (torch.randn((16, 256), generator=g) * 3.0).to(torch.bfloat16)
    x[0] = 0.0
    q, s, gs = oracle.quant_nvfp4(_bits(x))
    assert gs[0] == 1.0 and not q[0].any() and not s[0].any()       # all-zero row
    xf = x.float().numpy().astype(np.float64)
    for t in range(1, 16):
        assert gs[t] == np.float32(np.abs(xf[t]).max() / 2688.0)
        codes = np.stack([q[t] & 15, q[t] >> 4], 1).reshape(-1)
        val = np.array([oracle.e2m1_value(int(c)) for c in codes])
        sc = np.repeat([oracle.e4m3_value(int(b)) for b in s[t]], 16) * float(gs[t])
        # every element within half a grid step (at most 1 near 6, in units of the block scale)
        assert np.all(np.abs(val * sc - xf[t]) <= 1.0 * sc + 1e-12)
        # each block's largest element lands near the top of the E2M1 range
        blk = np.abs(xf[t]).reshape(-1, 16).max(1)
        assert np.all(np.abs(val.reshape(-1, 16)).max(1)[blk > 0] >= 4.0)
