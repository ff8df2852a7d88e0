"""moe_dispatch_no_workspace: the dispatch entry point for callers that cannot
allocate device memory (their memory is planned and owned by a host framework,
or cudaMalloc would stall a latency-critical loop), so it takes no workspace
and keeps its scratch tables in a fixed array inside the library.

It is checked through the C ABI against moe_dispatch (which uses a caller
workspace) on two different calls in a row, since every call reuses the same
built-in array.  This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import top_routing_expert_gate_b300 as moe
from top_routing_expert_gate_b300 import _binding as B

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _idx(T, E, k, seed, skew):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn((T, E), generator=g) - skew * torch.log(torch.arange(E) + 1.0)
    return torch.topk(z, k, dim=1).indices.to(torch.int32).contiguous().to(DEV)


def _outputs(cfg):
    E, A = cfg.n_experts, cfg.T * cfg.top_k
    return {"counts": torch.full((E,), -7, dtype=torch.int32, device=DEV),
            "drops": torch.full((E,), -7, dtype=torch.int32, device=DEV),
            "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
            "perm": torch.full((A,), -7, dtype=torch.int32, device=DEV),
            "drop_mask": torch.full((A,), 7, dtype=torch.uint8, device=DEV)}


def _no_workspace(cfg, idx):
    lib = B.load_library()
    o = _outputs(cfg)
    st = lib.moe_dispatch_no_workspace(
        ctypes.byref(cfg), idx.data_ptr(), o["counts"].data_ptr(), o["drops"].data_ptr(),
        o["offsets"].data_ptr(), o["perm"].data_ptr(), o["drop_mask"].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == B.MOE_OK, lib.moe_status_string(st)
    return o


def _with_workspace(cfg, idx):
    ws = moe.Workspace(cfg)
    o = _outputs(cfg)
    moe.moe_dispatch(cfg, idx, o["counts"], o["drops"], o["offsets"], o["perm"],
                     o["drop_mask"], ws)
    return o


def _assert_same(a, b, A):
    for key in ("counts", "drops", "offsets", "drop_mask"):
        assert torch.equal(a[key], b[key]), key
    n = int(a["offsets"][-1].item())
    assert torch.equal(a["perm"][:n], b["perm"][:n])
    assert int(a["counts"].sum() + a["drops"].sum()) == A


def test_no_workspace_dispatch_matches_workspace_dispatch_twice():
    # first call: DeepSeek-V3-sized routing (65536 assignments, 256 experts)
    # with a capacity that drops; second call: a different, smaller layer, so
    # leftovers from the first call in the shared array would show up.
    cases = [
        (moe.make_config(8192, 64, 256, 8, 128, capacity=200), 3, 1.0),
        (moe.make_config(3000, 64, 64, 1, 128, capacity=60), 4, 1.2),
    ]
    for cfg, seed, skew in cases:
        idx = _idx(cfg.T, cfg.n_experts, cfg.top_k, seed, skew)
        got = _no_workspace(cfg, idx)
        want = _with_workspace(cfg, idx)
        torch.cuda.synchronize()
        _assert_same(got, want, cfg.T * cfg.top_k)
        assert int(got["drops"].sum()) > 0


def test_no_workspace_dispatch_rejects_oversize_batch():
    lib = B.load_library()
    cfg = moe.make_config(131072 // 8 + 1, 64, 256, 8, 128)   # one token over the limit
    fake = 0x10000
    st = lib.moe_dispatch_no_workspace(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake,
                                       None)
    assert st == B.MOE_ERR_UNSUPPORTED


def test_no_workspace_dispatch_out_of_range_index_is_dropped():
    # With no status word, an expert index outside [0, E) is counted nowhere
    # and its assignment is marked dropped; the valid assignments dispatch as
    # moe_dispatch dispatches them (which also records the bad index in its
    # workspace status word).
    cfg = moe.make_config(1000, 64, 16, 2, 128, capacity=150)
    idx = _idx(cfg.T, cfg.n_experts, cfg.top_k, 5, 1.0)
    bad = [(3, 0, cfg.n_experts), (700, 1, -1)]      # (token, choice, index)
    for t, j, e in bad:
        idx[t, j] = e
    got = _no_workspace(cfg, idx)
    ws = moe.Workspace(cfg)
    want = _outputs(cfg)
    moe.moe_dispatch(cfg, idx, want["counts"], want["drops"], want["offsets"], want["perm"],
                     want["drop_mask"], ws)
    torch.cuda.synchronize()
    A = cfg.T * cfg.top_k
    for key in ("counts", "drops", "offsets", "drop_mask"):
        assert torch.equal(got[key], want[key]), key
    n = int(got["offsets"][-1].item())
    assert torch.equal(got["perm"][:n], want["perm"][:n])
    assert int(got["counts"].sum() + got["drops"].sum()) == A - len(bad)
    for t, j, _ in bad:
        assert int(got["drop_mask"][t * cfg.top_k + j].item()) == 1
        assert not bool((got["perm"][:n] == t * cfg.top_k + j).any())
    assert moe.moe_get_error(ws) == B.MOE_ERR_DEVICE
