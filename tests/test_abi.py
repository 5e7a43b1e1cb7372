"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function include/situ_moe.h declares, and rejects bad
arguments before launching anything."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from block_scaled_fp4_permute_gb300 import binding, build

HEADER = os.path.join(ROOT, "include", "situ_moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_header_declares_the_page_contract_calls():
    names = declared_functions()
    for n in ("situ_moe_permute", "situ_moe_quant_mxfp8", "situ_moe_forward",
              "situ_moe_workspace_size", "situ_moe_permute_workspace_size", "situ_status_string"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    raw = ctypes.CDLL(binding.library_path())
    for n in declared_functions():
        assert hasattr(raw, n), n


def _args(**over):
    a = dict(T=4, H=64, I=32, num_experts_total=8, num_local_experts=8, local_expert_offset=0,
             top_k=2, act_dtype=0, weight_dtype=0)
    a.update(over)
    s = binding.SituMoeArgs(**a)
    for f in ("hidden_states", "topk_ids", "topk_weights", "w1", "w1_scale", "w2", "w2_scale",
              "gemm1_alpha", "gemm1_beta", "out"):
        setattr(s, f, 0x1000)     # never dereferenced: validation fails first or T == 0
    return s


def _fwd(lib, args, ws=0x2000, nbytes=1 << 40):
    return lib.situ_moe_forward(ctypes.byref(args), ctypes.c_void_p(ws), nbytes, None)


@pytest.mark.parametrize("over,status", [
    (dict(H=48), 2), (dict(I=40), 2), (dict(top_k=17), 2), (dict(top_k=0), 2), (dict(T=-1), 2),
    (dict(local_expert_offset=4), 2), (dict(num_local_experts=0), 2),
    (dict(num_local_experts=5000, num_experts_total=6000), 2),
    (dict(act_dtype=1, weight_dtype=1), 3), (dict(act_dtype=0, weight_dtype=1), 3),
])
def test_forward_rejects_bad_shapes(lib, over, status):
    assert _fwd(lib, _args(**over)) == status


def test_forward_requires_situ_caps(lib):
    # the SiTU caps have no default (TensorRT-LLM PR #17865 requires non-null
    # swiglu_alpha / swiglu_beta for SiTU instead of a silent zero)
    a = _args()
    a.gemm1_beta = None
    assert _fwd(lib, a) == 1
    a = _args()
    a.gemm1_alpha = None
    assert _fwd(lib, a) == 1


def test_forward_other_errors(lib):
    a = _args()
    a.w1 = 0x1001
    assert _fwd(lib, a) == 6                         # misaligned
    assert _fwd(lib, _args(), nbytes=16) == 4        # workspace too small
    assert _fwd(lib, _args(), ws=0) == 1
    a = _args(act_dtype=1)                           # MXFP8 needs hidden_states_q / scale
    assert _fwd(lib, a) == 1
    assert _fwd(lib, _args(T=0)) == 0                # nothing to do, nothing launched


def test_device_status_argument_errors(lib):
    code = ctypes.c_int32(-1)
    assert lib.situ_moe_device_status(None, ctypes.c_void_p(16), None, ctypes.byref(code)) == 1
    assert code.value == 0
    assert lib.situ_moe_device_status(ctypes.byref(_args()), None, None, None) == 1
    assert lib.situ_moe_device_status(ctypes.byref(_args(top_k=0)), ctypes.c_void_p(16), None, None) == 2
    # T == 0: nothing ran, nothing to read
    assert lib.situ_moe_device_status(ctypes.byref(_args(T=0)), ctypes.c_void_p(16), None, None) == 0


def test_packed_scales_size_and_errors(lib):
    ok = _args(H=256, I=128)
    n = lib.situ_moe_packed_scales_size(ctypes.byref(ok))
    assert n > 0
    assert lib.situ_moe_packed_scales_size(ctypes.byref(_args(H=256, I=96))) == 0   # I % 128
    # NVFP4: two packings (H a multiple of 256, I of 128): the FC1 tiles, E_loc x
    # I/128 weight tiles x H/256 stages x 4 KB, then the FC2 tiles of a requantised
    # H1, E_loc x H/256 weight tiles x ceil(I/256) stages x 4 KB
    nv = lib.situ_moe_packed_scales_size(ctypes.byref(_args(H=512, I=256, act_dtype=2, weight_dtype=1)))
    assert nv == 8 * 2 * 2 * 4096 + 8 * 2 * 1 * 4096
    nv3 = lib.situ_moe_packed_scales_size(ctypes.byref(_args(H=512, I=384, act_dtype=2, weight_dtype=1)))
    assert nv3 == 8 * 3 * 2 * 4096 + 8 * 2 * 2 * 4096   # a half last stage of I counts whole
    assert lib.situ_moe_packed_scales_size(ctypes.byref(_args(H=384, I=128, act_dtype=2, weight_dtype=1))) == 0
    assert lib.situ_moe_packed_scales_size(None) == 0
    buf = ctypes.c_void_p(256)
    assert lib.situ_moe_pack_scales(None, buf, n, None) == 1
    assert lib.situ_moe_pack_scales(ctypes.byref(ok), None, n, None) == 1
    assert lib.situ_moe_pack_scales(ctypes.byref(_args(H=256, I=96)), buf, n, None) == 3
    assert lib.situ_moe_pack_scales(ctypes.byref(ok), ctypes.c_void_p(264), n, None) == 6
    assert lib.situ_moe_pack_scales(ctypes.byref(ok), buf, n - 1, None) == 4


def test_wait_selftest_argument_errors(lib):
    assert lib.situ_moe_wait_selftest(None, None) == 1
    assert lib.situ_moe_wait_selftest(ctypes.c_void_p(0x1002), None) == 6


def test_workspace_size_grows_with_tokens(lib):
    small = lib.situ_moe_workspace_size(ctypes.byref(_args(T=4)))
    big = lib.situ_moe_workspace_size(ctypes.byref(_args(T=400)))
    assert 0 < small < big
    assert lib.situ_moe_workspace_size(ctypes.byref(_args(top_k=0))) == 0


def test_permute_and_quant_validation(lib):
    vp = ctypes.c_void_p
    ok_ptr = vp(0x1000)
    assert lib.situ_moe_permute(ok_ptr, 4, 0, 8, 8, 0, ok_ptr, ok_ptr, ok_ptr, ok_ptr, ok_ptr,
                                1 << 20, None) == 2
    assert lib.situ_moe_permute(ok_ptr, 4, 2, 8, 8, 1, ok_ptr, ok_ptr, ok_ptr, ok_ptr, ok_ptr,
                                1 << 20, None) == 2
    assert lib.situ_moe_permute(ok_ptr, 4, 2, 8, 8, 0, ok_ptr, ok_ptr, ok_ptr, ok_ptr, ok_ptr,
                                0, None) == 4
    assert lib.situ_moe_permute(None, 4, 2, 8, 8, 0, ok_ptr, ok_ptr, ok_ptr, ok_ptr, ok_ptr,
                                1 << 20, None) == 1
    assert lib.situ_moe_permute(None, 0, 2, 8, 8, 0, None, None, None, None, None, 0, None) == 0
    assert lib.situ_moe_quant_mxfp8(ok_ptr, 4, 48, ok_ptr, ok_ptr, None) == 2
    assert lib.situ_moe_quant_mxfp8(None, 4, 64, ok_ptr, ok_ptr, None) == 1
    assert lib.situ_moe_quant_mxfp8(vp(0x1008), 4, 64, ok_ptr, ok_ptr, None) == 6
    assert lib.situ_moe_quant_mxfp8(None, 0, 64, None, None, None) == 0
    assert lib.situ_moe_permute_workspace_size(100, 16, 896) >= 4 * 896


def test_permute_noalloc_rejects_without_launch(lib):
    """Every rejection of the allocation-free permute returns before any
    CUDA call (the fake pointers are never dereferenced), so these run on
    the CPU: bad shapes, NULL and misaligned pointers, and a request beyond
    the fixed scratch (ceil(T*K/4096) * E_loc > SITU_NOALLOC_SCRATCH_INTS)."""
    vp = ctypes.c_void_p
    p = vp(0x1000)
    f = lib.situ_moe_permute_noalloc
    assert f(p, 4, 0, 8, 8, 0, p, p, p, p, None) == 2            # top_k 0
    assert f(p, 4, 17, 8, 8, 0, p, p, p, p, None) == 2           # top_k > 16
    assert f(p, -1, 2, 8, 8, 0, p, p, p, p, None) == 2           # T < 0
    assert f(p, 4, 2, 8, 8, 1, p, p, p, p, None) == 2            # shard beyond E_total
    assert f(p, 4, 2, 8, 0, 0, p, p, p, p, None) == 2            # no local expert
    assert f(None, 4, 2, 8, 8, 0, p, p, p, p, None) == 1
    assert f(p, 4, 2, 8, 8, 0, p, p, None, p, None) == 1
    assert f(vp(0x1004), 4, 2, 8, 8, 0, p, p, p, p, None) == 6
    assert f(p, 4, 2, 8, 8, 0, p, p, p, vp(0x1008), None) == 6
    assert f(p, 300_000, 16, 1024, 1024, 0, p, p, p, p, None) == 4
    assert f(None, 0, 2, 8, 8, 0, None, None, None, None, None) == 0   # T == 0: nothing


def test_route_topk_argument_errors(lib):
    vp = ctypes.c_void_p
    p = vp(0x1000)
    f = lib.situ_moe_route_topk
    assert f(p, 4, 8, 0, 1, p, p, None) == 2       # top_k 0
    assert f(p, 4, 8, 9, 1, p, p, None) == 2       # top_k > E
    assert f(p, 4, 32, 17, 1, p, p, None) == 2     # top_k > 16
    assert f(p, -1, 8, 2, 1, p, p, None) == 2
    assert f(p, 4, 0, 1, 1, p, p, None) == 2
    assert f(p, 4, 8, 2, 2, p, p, None) == 3       # renormalize not 0 / 1
    assert f(None, 4, 8, 2, 1, p, p, None) == 1
    assert f(p, 4, 8, 2, 1, p, None, None) == 1
    assert f(vp(0x1002), 4, 8, 2, 1, p, p, None) == 6
    assert f(None, 0, 8, 2, 1, None, None, None) == 0   # T == 0: nothing


def test_forward_wait_test_argument_errors(lib):
    f = lib.situ_moe_forward_wait_test
    a = _args(H=256, I=128)   # the block-scaled decode tiles
    assert f(None, ctypes.c_void_p(0x2000), 1 << 40, None, 0, 100) == 1
    assert f(ctypes.byref(a), ctypes.c_void_p(0x2000), 1 << 40, None, -1, 100) == 2
    assert f(ctypes.byref(a), ctypes.c_void_p(0x2000), 1 << 40, None, 0, 0) == 2
    assert f(ctypes.byref(a), ctypes.c_void_p(0x2000), 1 << 40, None, 0, 2000000) == 2
    assert f(ctypes.byref(_args()), ctypes.c_void_p(0x2000), 1 << 40, None, 0, 100) == 3   # register tiles
    bad = _args(H=256, I=128)
    bad.gemm1_beta = None
    assert f(ctypes.byref(bad), ctypes.c_void_p(0x2000), 1 << 40, None, 0, 100) == 1


def test_tc_peak_argument_errors(lib):
    vp = ctypes.c_void_p
    d = ctypes.c_double(0.0)
    assert lib.situ_tc_peak(0, 64, None, ctypes.byref(d), None) == 1
    assert lib.situ_tc_peak(0, 64, vp(0x1000), None, None) == 1
    assert lib.situ_tc_peak(0, 64, vp(0x1002), ctypes.byref(d), None) == 6
    assert lib.situ_tc_peak(3, 64, vp(0x1000), ctypes.byref(d), None) == 3
    assert lib.situ_tc_peak(0, 6, vp(0x1000), ctypes.byref(d), None) == 2
    assert lib.situ_tc_peak(0, 0, vp(0x1000), ctypes.byref(d), None) == 2


def test_status_strings(lib):
    for s in range(7):
        assert binding.status_string(s).startswith("SITU_")


def test_forward_launch_count(lib):
    n = lambda a: lib.situ_moe_forward_launches(ctypes.byref(a))
    # H, I not multiples of 128: decode-tile register path, one permute launch
    assert n(_args()) == 5
    # block-scaled decode tiles: permute, gather, FC1, FC2, combine, plus four
    # scale packings when the caller keeps no packed scales
    assert n(_args(H=256, I=128)) == 9
    packed = _args(H=256, I=128)
    packed.scales_packed = 0x4000
    assert n(packed) == 5
    # prefill routing (bf16): permute (one block), gather, FC1, H1 gather, FC2, combine
    assert n(_args(T=400, H=64, I=32)) == 6
    # block-scaled prefill (bf16 rows as hi + lo): permute, gather, FC1, FC2, combine;
    # fused combine: the combine becomes the accumulator's rounding, plus its zeroing
    pre = _args(T=400, H=256, I=128)
    pre.scales_packed = 0x4000
    assert n(pre) == 5
    pre.fuse_combine = 1
    assert n(pre) == 6
    # NVFP4 tiles: permute, gather, FC1 (mxf4nvf4), H1 to f16, FC2 (weights expanded to f16 in
    # TMEM, kind::f16), combine, plus one scale packing
    nv = _args(H=256, I=128, act_dtype=2, weight_dtype=1)
    for f in ("hidden_states_q", "hidden_states_scale", "hidden_states_gscale", "w1_gscale", "w2_gscale"):
        setattr(nv, f, 0x1000)
    assert n(nv) == 7
    nv.scales_packed = 0x4000
    assert n(nv) == 6
    assert n(_args(T=0)) == 0
    bad = _args()
    bad.gemm1_alpha = None
    assert n(bad) == -1
    assert lib.situ_moe_forward_launches(None) == -1


@pytest.mark.parametrize("T,launches", [
    (50, 7),     # 12.5 rows per expert: 16-token tiles, one tile table, H1 to f16 for the FC2
    (100, 7),    # 25: both GEMMs on 64-token tiles, still one tile table
    (300, 7),    # 75: FC2 on 128-token tiles of a second tile table
    (2048, 7),   # 512: the widest routing still on the NVFP4 tiles (4,096 slots, one permute launch)
    (2056, 8),   # 514: the f16 prefill tiles, and three permute launches from 4,097 slots on
])
def test_nvfp4_path_choice_by_rows_per_expert(lib, T, launches):
    """The host picks the NVFP4 kernels from T * top_k / E_total alone:
    per-launch counts pin the 16 / 64 / 128-token tile thresholds and the
    hand-over to the f16 prefill tiles above 512 rows per expert."""
    a = _args(T=T, H=256, I=128, num_experts_total=8, num_local_experts=8, top_k=2, act_dtype=2,
              weight_dtype=1)
    for f in ("hidden_states_q", "hidden_states_scale", "hidden_states_gscale", "w1_gscale", "w2_gscale"):
        setattr(a, f, 0x1000)
    assert lib.situ_moe_forward_launches(ctypes.byref(a)) == launches


@pytest.mark.parametrize("T,fuse,w1,launches", [
    (24, 1, 0x1000, 5),   # 6 rows per expert: block-scaled decode tiles (no fused combine there)
    (28, 1, 0x1000, 6),   # 7: block-scaled prefill tiles, combine fused (+ accumulator zeroing)
    (28, 0, 0x1000, 5),   # 7: block-scaled prefill tiles, separate combine
    (24, 0, 0x1010, 5),   # W1 not 32-byte aligned: no 4-bit tensor map; decode register tiles
    (28, 0, 0x1010, 6),   # ... and above 6 rows per expert the f16 prefill tiles (+ H1 gather)
])
def test_mxfp4_path_choice(lib, T, fuse, w1, launches):
    """MXFP4 weights with H, I multiples of 128: up to six rows per expert the
    decode tiles, above them the prefill tiles; weights the 4-bit tensor maps
    cannot address (base not 32-byte aligned) take the register / f16 paths."""
    a = _args(T=T, H=256, I=128, num_experts_total=8, num_local_experts=8, top_k=2)
    a.scales_packed = 0x4000
    a.fuse_combine = fuse
    a.w1 = w1
    assert lib.situ_moe_forward_launches(ctypes.byref(a)) == launches


def test_quant_nvfp4_argument_errors(lib):
    p = ctypes.c_void_p(256)
    assert lib.situ_moe_quant_nvfp4(p, 4, 40, p, p, p, None) == 2     # H % 16
    assert lib.situ_moe_quant_nvfp4(p, -1, 64, p, p, p, None) == 2
    assert lib.situ_moe_quant_nvfp4(p, 0, 64, None, None, None, None) == 0
    assert lib.situ_moe_quant_nvfp4(None, 4, 64, p, p, p, None) == 1
    assert lib.situ_moe_quant_nvfp4(ctypes.c_void_p(264), 4, 64, p, p, p, None) == 6


def test_forward_tactic_field(lib):
    # TokenSpeed SiTU's runtime API: tactic = (-1, -1) is the first valid
    # configuration; this library has one per shape, selected by -1 or 0
    for t in ((-1, -1), (0, 0), (-1, 0)):
        a = _args()
        a.tactic[0], a.tactic[1] = t
        assert lib.situ_moe_forward_launches(ctypes.byref(a)) == 5
    for t in ((1, -1), (-1, 2), (-2, -1)):
        a = _args()
        a.tactic[0], a.tactic[1] = t
        assert _fwd(lib, a) == 3


def _nv_args(**over):
    a = _args(**{**dict(H=256, I=128, act_dtype=2, weight_dtype=1), **over})
    for f in ("hidden_states_q", "hidden_states_scale", "hidden_states_gscale", "w1_gscale", "w2_gscale"):
        setattr(a, f, 0x1000)
    return a


def test_h1_nvfp4_option(lib):
    """The requantised NVFP4 H1 belongs to the NVFP4 chain on its tile shapes:
    one more launch (the requantisation), plus the FC2 scale packing when the
    call packs its own scales; the 128-token FC2 tile table is not needed."""
    n = lambda a: lib.situ_moe_forward_launches(ctypes.byref(a))
    a = _nv_args()
    a.h1_nvfp4 = 1
    assert n(a) == 8                      # permute, 2 packings, gather, FC1, requant, FC2, combine
    a.scales_packed = 0x4000
    assert n(a) == 6
    wide = _nv_args(T=300, num_experts_total=8, num_local_experts=8, top_k=2)
    wide.scales_packed = 0x4000
    assert n(wide) == 6                   # 64-token tiles, 75 rows per expert: the second table
    wide.h1_nvfp4 = 1                     # (fcv's 128-token tiles) is left out
    assert n(wide) == 6
    f16 = _nv_args(T=2056, num_experts_total=8, num_local_experts=8, top_k=2)
    f16.h1_nvfp4 = 1
    assert n(f16) == 9                    # f16 prefill tiles: + the requantisation
    for bad in (_args(), _args(H=256, I=128)):   # MXFP4 pairs
        bad.h1_nvfp4 = 1
        assert _fwd(lib, bad) == 3
    odd = _nv_args(H=384)                 # H not a multiple of 256
    odd.h1_nvfp4 = 1
    assert _fwd(lib, odd) == 3
    two = _nv_args()
    two.h1_nvfp4 = 2
    assert _fwd(lib, two) == 3


def test_forward_rejects_unknown_activation(lib):
    a = _args()
    a.activation = 2
    assert _fwd(lib, a) == 3
    assert lib.situ_moe_forward_launches(ctypes.byref(a)) == -1
