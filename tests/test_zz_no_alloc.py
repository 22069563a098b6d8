"""The allocation-free dispatch entry point matches the workspace one (GPU).

lrm_dispatch_permute_noalloc serves callers that cannot allocate device
memory (a plugin handed only its tensors, or a host whose memory manager
owns the device budget): its scratch is built into the library. This file
is collected last on purpose, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from workloads import generate, get_config

pytestmark = pytest.mark.gpu


def _buffers(N, E, dev):
    i32 = torch.int32
    return (torch.empty(max(N, 1), dtype=i32, device=dev),
            torch.empty(max(N, 1), dtype=i32, device=dev),
            torch.empty(E, dtype=i32, device=dev), torch.empty(E + 1, dtype=i32, device=dev))


def _reference(lrm, shape, idx, N, E, dev):
    ws_bytes = lrm.lrm_workspace_bytes(shape)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    perm, inv, counts, off = _buffers(N, E, dev)
    lrm.lrm_dispatch_permute(shape, idx, perm, inv, counts, off, ws, ws_bytes)
    return perm, inv, counts, off


@pytest.mark.parametrize("name,over", [
    ("qwen3-30b-a3b-t4k", {}),                      # 32768 pairs: one cluster, no table
    ("stress-e256", {"D": 64, "H": 64}),            # 262144 pairs, 256 experts: the tables
    ("tiny", {}),
])
def test_noalloc_dispatch_matches_workspace_dispatch_twice(name, over):
    from demand_side_expert_gb300 import lrm

    dev = torch.device("cuda:0")
    cfg = get_config(name, **over)
    N, E = cfg.N, cfg.E
    shape = lrm.make_shape(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, lrm.LRM_BF16)
    inputs = [generate(cfg, device=dev, seed=s)["topk_idx"] for s in (0, 1)]
    for idx in inputs:  # two calls in a row on different routings
        ref = _reference(lrm, shape, idx, N, E, dev)
        got = _buffers(N, E, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lrm.lrm_dispatch_permute_noalloc(shape, idx, *got, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for a, b, n in zip(ref, got, (N, N, E, E + 1)):
            assert torch.equal(a[:n], b[:n])


def test_noalloc_dispatch_with_1000_experts():
    """1000 experts and 133,120 pairs (65 chunks, above the single-launch
    limit): the count and scatter kernels need more than 48 KiB of shared
    memory, so the call first raises their limit; the result is the workspace
    dispatch's bit for bit, twice."""
    from demand_side_expert_gb300 import lrm

    dev = torch.device("cuda:0")
    cfg = get_config("qwen3-30b-a3b-t4k", T=16640, D=64, H=64, E=1000, K=8)
    N, E = cfg.N, cfg.E
    shape = lrm.make_shape(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, lrm.LRM_BF16)
    idx = generate(cfg, device=dev)["topk_idx"]
    ref = _reference(lrm, shape, idx, N, E, dev)
    for _ in range(2):
        got = _buffers(N, E, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lrm.lrm_dispatch_permute_noalloc(shape, idx, *got, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for a, b, n in zip(ref, got, (N, N, E, E + 1)):
            assert torch.equal(a[:n], b[:n])


def test_noalloc_dispatch_allocates_no_device_memory():
    """After a first call (which may load the kernels and look up the
    scratch array's address), further calls leave the device's free memory
    and PyTorch's allocator untouched."""
    from demand_side_expert_gb300 import lrm

    dev = torch.device("cuda:0")
    cfg = get_config("stress-e256", D=64, H=64)
    N, E = cfg.N, cfg.E
    shape = lrm.make_shape(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, lrm.LRM_BF16)
    idx = generate(cfg, device=dev)["topk_idx"]
    got = _buffers(N, E, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lrm.lrm_dispatch_permute_noalloc(shape, idx, *got, err)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for _ in range(3):
        lrm.lrm_dispatch_permute_noalloc(shape, idx, *got, err)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert int(err.item()) == 0


def test_noalloc_flags_bad_ids_like_the_workspace_path():
    from demand_side_expert_gb300 import lrm

    dev = torch.device("cuda:0")
    cfg = get_config("tiny")
    shape = lrm.make_shape(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, lrm.LRM_F32)
    idx = generate(cfg, device=dev)["topk_idx"].clone()
    idx[7, 1] = cfg.E + 3
    got = _buffers(cfg.N, cfg.E, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lrm.lrm_dispatch_permute_noalloc(shape, idx, *got, err)
    ref = _reference(lrm, shape, idx, cfg.N, cfg.E, dev)
    torch.cuda.synchronize()
    assert int(err.item()) & lrm.LRM_DEVERR_EXPERT_ID
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from demand_side_expert_gb300 import lrm

    # 1024 experts x 128 chunks of 2048 pairs exceeds the built-in tables
    shape = lrm.make_shape(32768, 64, 64, 1024, 8, lrm.LRM_BF16)
    status = lrm._lib.lrm_dispatch_permute_noalloc(ctypes.byref(shape), 256, 256, 256, 256,
                                                   256, None, None)
    assert status == lrm.LRM_ERR_WORKSPACE
    assert 1024 * 128 > lrm.LRM_NOALLOC_MAX_CHUNK_ENTRIES
    assert np.int64(256) * 128 <= lrm.LRM_NOALLOC_MAX_CHUNK_ENTRIES  # the stress layer fits
