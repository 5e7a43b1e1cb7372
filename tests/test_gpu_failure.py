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
