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
    # call 1: the Kimi-K3 prefill routing (131,072 slots, 896 local experts;
    # the three-launch count / scan / scatter path)
    cfg = W.CONFIGS["prefill_w4a8"]
    ids1, _ = W.routing(cfg["T"], cfg["K"], cfg["E_total"], cfg["routing"], 0)
    _both(ids1, cfg["E_total"], cfg["E_loc"], cfg["off"])
    # call 2 right after: a smaller EP-shard routing with out-of-range IDs,
    # on the scratch the first call left behind
    rng = np.random.default_rng(7)
    ids2 = rng.integers(-2, 900, (3000, 16)).astype(np.int32)
    counts, offsets, psrc, s2r = _both(ids2, 896, 112, 336)
    assert int(offsets[-1]) == int(((ids2 >= 336) & (ids2 < 448)).sum())


def test_decode_routing_single_launch_path():
    # the Kimi-K3 decode routing (1,024 slots, 896 local experts) takes the
    # one-CTA permute, twice in a row, and a strided view of a wider routing
    # tensor is read as its own elements
    cfg = W.CONFIGS["decode"]
    ids, _ = W.routing(cfg["T"], cfg["K"], cfg["E_total"], cfg["routing"], 3)
    _both(ids, cfg["E_total"], cfg["E_loc"], cfg["off"])
    _both(ids[::-1].copy(), cfg["E_total"], cfg["E_loc"], cfg["off"])
    wide = torch.from_numpy(np.concatenate([ids, ids + 1], axis=1)).cuda()
    view = wide[:, :cfg["K"]]
    assert not view.is_contiguous()
    got = binding.situ_moe_permute_noalloc(view, cfg["E_total"], cfg["E_loc"], cfg["off"])
    ref = binding.situ_moe_permute(torch.from_numpy(ids).cuda(), cfg["E_total"], cfg["E_loc"], cfg["off"])
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
