"""Device-side failure detection without faulting the GPU.

A kernel whose bounded wait can never be satisfied must give up after its
limit, report MOE_ERR_TIMEOUT through the workspace status word, and leave
the CUDA context usable for the next layer call.  Host-side argument checks
are covered (without a GPU) in test_abi.py.
"""

import time

import pytest
import torch

import top_routing_expert_gate_b300 as moe
from top_routing_expert_gate_b300 import _binding as B
from workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    s = MoEShape("after", T=96, d=128, E=4, k=2, F=128, F_s=0, gate="softmax",
                 renormalize=True, rsf=1.0, capacity_factor=None, zipf_s=None, dtype="bf16")
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    lib = B.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert lib.moe_selftest_bounded_wait(ws.ptr, ws.nbytes, 20_000_000, stream) == B.MOE_OK
    assert moe.moe_get_error(ws) == B.MOE_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 5.0, elapsed          # it waited about 20 ms, then returned
    assert moe.moe_get_error(ws) == B.MOE_OK       # reading cleared the status word
    # the context still works: a full layer call afterwards runs and is sane
    inp = make_inputs(s, device="cuda", seed=0)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == B.MOE_OK
    assert torch.isfinite(out["y"]).all()
    assert int(out["counts"].sum()) == s.T * s.k


def test_selftest_rejects_bad_limits():
    lib = B.load_library()
    cfg = moe.make_config(8, 64, 4, 2, 128)
    ws = moe.Workspace(cfg)
    assert lib.moe_selftest_bounded_wait(ws.ptr, ws.nbytes, 0, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(ws.ptr, ws.nbytes, 5_000_000_000, None) == \
        B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(None, 0, 1000, None) == B.MOE_ERR_WORKSPACE


def test_out_of_range_permutation_is_reported_not_read():
    # moe_grouped_swiglu takes the caller's permutation.  A grouped row naming
    # an assignment past the batch is recorded in the status word
    # (MOE_ERR_DEVICE) and the gather skips it, reading nothing outside x; the
    # next call on the same workspace is clean.
    s = MoEShape("bad_perm", T=96, d=128, E=4, k=2, F=128, F_s=0, gate="softmax",
                 renormalize=True, rsf=1.0, capacity_factor=None, zipf_s=None, dtype="bf16")
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    inp = make_inputs(s, device="cuda", seed=3)
    w = moe.LayerWeights.from_inputs(inp)
    r = moe.route(cfg, inp["x"], w.w_router, None, ws=ws)
    dsp = moe.dispatch(cfg, r["topk_idx"], ws=ws)
    A = s.T * s.k
    bad = dsp["perm"].clone()
    bad[5] = A + 1000
    y_perm = torch.empty((A, s.d), dtype=torch.float32, device="cuda")
    moe.moe_grouped_swiglu(cfg, inp["x"], bad, dsp["offsets"], w.w_gate, w.w_up, w.w_down,
                           None, None, None, y_perm, None, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == B.MOE_ERR_DEVICE
    moe.moe_grouped_swiglu(cfg, inp["x"], dsp["perm"], dsp["offsets"], w.w_gate, w.w_up,
                           w.w_down, None, None, None, y_perm, None, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == B.MOE_OK
    assert torch.isfinite(y_perm[:A]).all()
