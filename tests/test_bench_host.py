"""The bench's roofline arithmetic on the CPU: the algorithmic bytes and
FLOPs that every bench line divides by, and the MMA kind (hence the peak)
each GEMM is judged against, recomputed by hand from the workload's shape."""
import os
import sys
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _wl(T, H, I, E, K, act, wt, E_loc=None):
    return SimpleNamespace(T=T, H=H, I=I, E_total=E, E_loc=E if E_loc is None else E_loc, K=K, act=act, wt=wt)


def test_decode_layer_bytes_by_hand():
    """Kimi-K3 TP8 decode, w4a16: each touched expert's MXFP4 W1 is
    2I x H/2 code bytes plus 2I x H/32 scale bytes (1,462,272 B), W2 is
    H x I/2 + H x I/32 (731,136 B); the layer adds the bf16 input and output
    once and 8 bytes of routing per slot.  603 of 896 experts are touched by
    the seed-0 routing, which gives the 1,323,550,720 bytes of the bench line."""
    wl = _wl(64, 3584, 384, 896, 16, act=0, wt=0)
    R, touched = 1024, 603
    b = bench.algorithmic_bytes(wl, R, touched)
    w1, w2 = 603 * 1_462_272, 603 * 731_136
    assert b["layer"] == w1 + w2 + 64 * 3584 * 2 + 64 * 16 * 8 + 64 * 3584 * 2 == 1_323_550_720
    # FC1 reads its weights, the bf16 rows as hi + lo E4M3 (2H bytes) and writes H1 (2I bytes per row)
    assert b["fc1"] == w1 + R * 2 * 3584 + R * 2 * 384
    # the gather reads the input once and writes the expert-ordered rows once
    assert b["gather"] == 64 * 3584 * 2 + R * 2 * 3584
    # FC2 writes fp32 Y rows on the decode tiles, which the combine reads back
    assert b["fc2"] == w2 + R * 2 * 384 + R * 3584 * 4
    assert b["combine"] == R * 3584 * 4 + 64 * 16 * 8 + 64 * 3584 * 2


def test_prefill_w4a8_bytes_by_hand():
    """Kimi-K3 TP8 prefill, w4a8: MXFP8 rows are H code bytes plus H/32
    scale bytes, H1 is MXFP8 (I + I/32 bytes per row), and the block-scaled
    prefill tiles write Y as f16 with one scale byte per 32 columns."""
    wl = _wl(8192, 3584, 384, 896, 16, act=1, wt=0)
    R, touched = 131072, 896
    b = bench.algorithmic_bytes(wl, R, touched)
    x_row = 3584 + 3584 / 32
    assert b["gather"] == 8192 * x_row + R * x_row
    assert b["fc2"] == 896 * (3584 * 384 // 2 + 3584 * 384 // 32) + R * (384 + 384 / 32) + R * 3584 * (2 + 1 / 32)
    assert b["quant"] == 8192 * 3584 * 2 + 8192 * 3584 + 8192 * 3584 // 32


def test_layer_flops_by_hand():
    wl = _wl(8192, 3584, 384, 896, 16, act=1, wt=0)
    # FC1: 2 R H (2I); FC2: 2 R I H
    assert bench.layer_flops(wl, 131072) == 2.0 * 131072 * 3584 * 768 + 2.0 * 131072 * 384 * 3584


def test_gemm_kinds_follow_the_path_choice():
    """The MXFP4 shapes run both GEMMs on kind::mxf8f6f4; the NVFP4 tiles
    (at most 512 rows per expert) run FC1 on kind::mxf4nvf4 and FC2 on bf16
    H1 (kind::f16), or on kind::mxf4nvf4 with H1 requantised; beyond 512 rows
    per expert, and for odd shapes, the f16 tiles."""
    assert bench.gemm_kinds(_wl(64, 3584, 384, 896, 16, 0, 0)) == {"fc1": "mxf8f6f4", "fc2": "mxf8f6f4"}
    assert bench.gemm_kinds(_wl(8192, 3584, 384, 896, 16, 1, 0)) == {"fc1": "mxf8f6f4", "fc2": "mxf8f6f4"}
    assert bench.gemm_kinds(_wl(256, 3584, 384, 896, 16, 2, 1)) == {"fc1": "mxf4nvf4", "fc2": "bf16"}
    assert bench.gemm_kinds(_wl(256, 3584, 384, 896, 16, 2, 1), h1_nvfp4=True) == {"fc1": "mxf4nvf4",
                                                                                    "fc2": "mxf4nvf4"}
    # 16384 x 16 / 896 = 292.6 rows per expert: still the NVFP4 tiles
    assert bench.gemm_kinds(_wl(16384, 3584, 384, 896, 16, 2, 1))["fc1"] == "mxf4nvf4"
    # 32768 x 16 / 896 = 585 rows per expert: the f16 tiles
    assert bench.gemm_kinds(_wl(32768, 3584, 384, 896, 16, 2, 1)) == {"fc1": "f16", "fc2": "f16"}
    # an H that is not a multiple of 128 leaves the block-scaled MXFP4 path
    assert bench.gemm_kinds(_wl(64, 3600, 384, 896, 16, 0, 0)) == {"fc1": "f16", "fc2": "f16"}


def test_tensor_peak_of_uses_the_measured_kind():
    tc = {"mxf8f6f4": {"tflops": 4868.0}, "mxf4nvf4": {"tflops": 9737.0}, "_source": "test"}
    assert bench.tensor_peak_of("mxf8f6f4", tc)[0] == 4868.0
    assert bench.tensor_peak_of("mxf4nvf4", tc)[0] == 9737.0
    bf16, _ = bench.tensor_peak_of("bf16", tc)
    assert bench.tensor_peak_of("f16", tc)[0] == bf16
    # no microbenchmark result for the kind: twice the bf16 figure, and it says so
    v, src = bench.tensor_peak_of("mxf8f6f4", None)
    assert v == 2.0 * bf16 and "nominal" in src
