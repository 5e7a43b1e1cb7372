"""The allocation-free permute entry point.

Some callers cannot allocate device memory where they route tokens, for
example an engine that owns all device memory through its own pool, or
code where a cudaMalloc would synchronise the device.  For them
situ_moe_permute_noalloc keeps its scratch in a fixed array inside the
library.  This test calls it through the C ABI twice in a row, on two
different routings, and checks each result bit for bit against the
workspace-taking situ_moe_permute (the permute's parity bar is exactness).
The second call sees the array as the first call left it.  The file is
collected last, so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp4_permute_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


def _both(ids_np, E_total, E_loc, off):
    ids = torch.from_numpy(ids_np).cuda()
    ref = binding.situ_moe_permute(ids, E_total, E_loc, off)
    got = binding.situ_moe_permute_noalloc(ids, E_total, E_loc, off)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    return got


def test_two_calls_match_the_workspace_permute():
    # call 1: the Kimi-K3 prefill routing (131,072 slots, 896 local experts)
    cfg = W.CONFIGS["prefill_w4a8"]
    ids1, _ = W.routing(cfg["T"], cfg["K"], cfg["E_total"], cfg["routing"], 0)
    _both(ids1, cfg["E_total"], cfg["E_loc"], cfg["off"])
    # call 2 right after: a smaller EP-shard routing with out-of-range IDs,
    # on the scratch the first call left behind
    rng = np.random.default_rng(7)
    ids2 = rng.integers(-2, 900, (3000, 16)).astype(np.int32)
    counts, offsets, psrc, s2r = _both(ids2, 896, 112, 336)
    assert int(offsets[-1]) == int(((ids2 >= 336) & (ids2 < 448)).sum())


def test_too_large_request_is_rejected_without_launch():
    # ceil(T*K/4096) * E_loc > SITU_NOALLOC_SCRATCH_INTS (1 << 20)
    T, K, E = 300_000, 16, 1024
    ids = torch.zeros((1, K), dtype=torch.int32, device="cuda")   # never read
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    st = binding.lib().situ_moe_permute_noalloc(
        binding._p(ids), T, K, E, E, 0, binding._p(dummy), binding._p(dummy),
        binding._p(dummy), binding._p(dummy), binding._stream(None))
    assert st == 4          # SITU_ERR_WORKSPACE_TOO_SMALL
