"""The failure path on the GPU, without a fault: a bounded device wait is
made to run out, and the CUDA context stays usable.

Every wait of the tensor-core GEMM kernels on their asynchronous copies and
MMAs is bounded (200 ms of the GPU's global timer); one that runs out records
a code in a status word and the kernel returns.  situ_moe_wait_selftest runs
that same wait on a barrier phase that nothing completes.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_permute_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


def test_bounded_wait_runs_out_and_reports_its_code():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.situ_moe_wait_selftest(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == binding.SITU_SELFTEST_WAIT_CODE
    assert 0.15 < waited < 30.0     # the wait gave up at its limit, it did not hang


def test_context_stays_usable_after_the_wait_ran_out():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.situ_moe_wait_selftest(status)
    torch.cuda.synchronize()
    assert int(status.item()) == binding.SITU_SELFTEST_WAIT_CODE
    # a whole layer on the tensor-core decode tiles, against the oracle
    wl = W.make("tiny", device="cuda")
    layer = binding.Layer(wl)
    out = layer().float().cpu().numpy()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ref = oracle.moe_forward(**W.oracle_kwargs(wl))
    rms = float(np.sqrt(np.mean(ref ** 2)))
    a = np.abs(ref)
    half_ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)
    assert float(np.max(np.abs(out - ref) - half_ulp)) <= 2e-2 * rms


def _parity(out, ref):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    a = np.abs(ref)
    half_ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)
    assert float(np.max(np.abs(out - ref) - half_ulp)) <= 2e-2 * rms


@pytest.mark.parametrize("skip_stage", [0, 1, 5, 12])
def test_gemm_gives_up_a_stage_that_never_lands_and_unwinds(skip_stage):
    """The FC1 GEMM's own failure path: CTA 0's producer leaves one K stage
    unissued, so the MMA issuer's bounded wait for it runs out (20 ms here).
    The call reports SITU_ERR_DEVICE_TIMEOUT through the status word with the
    code of the first wait that ran out -- the epilogue's wait for the
    accumulator (46), which starts first, or the MMA issuer's wait for the
    stage (43) -- and returns within a few limits; a normal forward
    on the same workspace then matches the oracle, so the kernel drained its
    copies and MMAs and released its tensor memory."""
    # the block-scaled decode tiles with more work items than CTAs: 64 experts x
    # 4 FC1 weight tiles, 8 K stages each, so CTA 0 runs two items (16 stages)
    wl = W.make("tiny", device="cuda", T=96, H=1024, I=512, E_total=64, E_loc=64, off=0, K=4,
                params="k3_random")
    layer = binding.Layer(wl)
    ref = oracle.moe_forward(**W.oracle_kwargs(wl))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.situ_moe_forward_wait_test(layer.args, layer.workspace, skip_stage, 20000)
    code = layer.device_status()
    waited = time.perf_counter() - t0
    assert code in (43, 46), code
    assert waited < 10.0
    for _ in range(2):
        out = layer().float().cpu().numpy()
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        _parity(out, ref)
