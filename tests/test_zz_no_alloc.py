"""The allocation-free permutation entry point gives the same results as the
workspace one.

moe_permute_noalloc serves callers that cannot hand the library a workspace
because they may not allocate device memory themselves (a serving engine that
owns every byte of device memory through its own allocator or budget, or a
latency-critical loop where a cudaMalloc and its possible device
synchronisation are not allowed).  Its scratch is a fixed array inside the
library, shared by every call.  This file is collected last so that a run
stopping at its first failure has already run every other test; it also
passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import top_routed_expert_gb300 as moe
from top_routed_expert_gb300 import abi

pytestmark = pytest.mark.gpu


def _ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E - 2, size=k, replace=False) for _ in range(T)]).astype(np.int32)


def _permute_both(T, E, k, seed):
    dev = "cuda"
    cfg = abi.make_config(T, 128, E, k, 64, 64)
    ids = torch.from_numpy(_ids(T, E, k, seed)).to(dev)
    out = []
    for use_ws in (True, False):
        offs = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
        sp = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
        row_of = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
        if use_ws:
            ws = torch.empty(abi.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
            abi.moe_permute(cfg, ids, offs, sp, row_of, ws)
        else:
            abi.moe_permute_noalloc(cfg, ids, offs, sp, row_of)
        assert abi.moe_get_device_status() == 0
        out.append((offs.cpu().numpy(), sp.cpu().numpy(), row_of.cpu().numpy()))
    return out


def test_noalloc_permute_matches_workspace_permute_twice():
    moe.build()
    abi.load()
    # two calls in a row: the second reuses the scratch the first left behind
    for T, E, k, seed in ((8192, 128, 8, 1), (3001, 128, 6, 2)):
        (o1, s1, r1), (o2, s2, r2) = _permute_both(T, E, k, seed)
        assert np.array_equal(o1, o2)       # integer results: bit-exact
        assert np.array_equal(s1, s2)
        assert np.array_equal(r1, r2)
        assert o1[-1] == T * k


def test_noalloc_permute_rejects_oversize():
    cfg = abi.make_config(abi.MOE_NOALLOC_MAX_PAIRS // 8 + 1, 128, 128, 8, 64, 64)
    dev = "cuda"
    dummy = torch.empty(16, dtype=torch.int32, device=dev)
    with pytest.raises(abi.MoEError) as ei:
        abi.moe_permute_noalloc(cfg, dummy, dummy, dummy, dummy)
    assert ei.value.code == 2      # MOE_ERR_UNSUPPORTED, before any launch
