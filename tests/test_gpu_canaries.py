"""Out-of-bounds writes, found without a sanitizer: the layer's output and
its workspace sit inside larger buffers whose margins hold a known byte
pattern, and after a forward on each GEMM path the margins must be intact
(and the result still matches the oracle)."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_permute_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu
PAD = 4096            # bytes of margin on each side (keeps 256-byte alignment)
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


def _oracle(wl):
    if wl.act == W.ACT_MXFP8:
        q, s = oracle.quant_mxfp8(wl.host("x_bf16"))
        kw = W.oracle_kwargs(wl, x_q=q, x_scale=s)
    elif wl.act == W.ACT_NVFP4:
        q, s, g = oracle.quant_nvfp4(wl.host("x_bf16"))
        kw = W.oracle_kwargs(wl, x_q=q, x_scale=s, x_gscale=g)
    else:
        kw = W.oracle_kwargs(wl)
    return oracle.moe_forward(**kw)


@pytest.mark.parametrize("over,fuse", [
    (dict(T=64, H=256, I=128, E_total=64, E_loc=64, off=0, K=4), False),              # block-scaled decode tiles
    (dict(T=64, H=256, I=128, E_total=64, E_loc=48, off=8, K=4, act=W.ACT_NVFP4,
          wt=W.W_NVFP4), False),                                                    # NVFP4 tiles, 16 tokens
    (dict(T=600, H=256, I=128, E_total=16, E_loc=16, off=0, K=2, act=W.ACT_NVFP4,
          wt=W.W_NVFP4), False),                                                    # NVFP4, 64 / 128 tokens
    (dict(T=300, H=256, I=128, E_total=4, E_loc=4, off=0, K=2, act=W.ACT_MXFP8), False),   # block-scaled prefill
    (dict(T=300, H=256, I=128, E_total=4, E_loc=4, off=0, K=2, act=W.ACT_MXFP8), True),    # ... fused combine
    (dict(T=257, H=640, I=256, E_total=6, E_loc=3, off=2, K=3), False),               # bf16 hi + lo prefill
    (dict(T=17, H=160, I=96, E_total=12, E_loc=5, off=4, K=3), False),                # register decode tiles
    (dict(T=29, H=320, I=160, E_total=16, E_loc=8, off=8, K=4, act=W.ACT_NVFP4,
          wt=W.W_NVFP4), False),                                                    # f16 prefill tiles
])
def test_margins_of_output_and_workspace_stay_intact(over, fuse):
    wl = W.make("tiny", device="cuda", params="k3_random", **over)
    n_out = wl.T * wl.H * 2
    out_buf = torch.full((n_out + 2 * PAD,), CANARY, dtype=torch.uint8, device="cuda")
    out = out_buf[PAD:PAD + n_out].view(torch.bfloat16).view(wl.T, wl.H)
    layer = binding.Layer(wl, out=out, fuse_combine=fuse)
    n_ws = layer.workspace.numel()
    ws_buf = torch.full((n_ws + 2 * PAD,), CANARY, dtype=torch.uint8, device="cuda")
    layer.workspace = ws_buf[PAD:PAD + n_ws]
    res = layer().float().cpu().numpy()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    for buf, n in ((out_buf, n_out), (ws_buf, n_ws)):
        head = buf[:PAD].cpu().numpy()
        tail = buf[PAD + n:].cpu().numpy()
        assert np.all(head == CANARY) and np.all(tail == CANARY), str(over)
    ref = _oracle(wl)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    a = np.abs(ref)
    half_ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)
    assert float(np.max(np.abs(res - ref) - half_ulp)) <= 2e-2 * rms, str(over)
