"""Failure detection without a GPU fault: the bounded waits of the scan's
lookback and of the fused layout + offsets kernel's grid barrier.

The workspace's tile counter is set to 1 from the host before a call, so
the block that should take tile 0 is handed an out-of-range tile instead
(and reports MP_ERR_INVALID_ARG) and tile 0 never publishes.  The other
tiles of source rank 0 then wait on a flag that nothing sets; each wait is
bounded (about a second), so the call must finish with MP_ERR_TIMEOUT in
the device error word, and the context must stay usable: a normal call on a
re-zeroed workspace right after gives the exact answer.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from combine_mp_layout_gb300 import binding as B
from combine_mp_layout_gb300 import workloads as wl
from combine_mp_layout_gb300.pipeline import EPPlan

pytestmark = pytest.mark.gpu


def test_lookback_wait_times_out_and_context_survives():
    inp = wl.make_ep(dict(R=2, N=1024, E=8, K=2, H=64, routing="uniform", dtype="bf16"), seed=1)
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H)
    plan.load(inp)
    B.check(plan.layout())
    torch.cuda.synchronize()
    # host-side injection: the first tile handed out is tile 1, not tile 0
    plan.workspace[:4].copy_(torch.tensor([1, 0, 0, 0], dtype=torch.uint8))
    plan.dev_err.zero_()
    t0 = time.time()
    B.check(plan.dispatch_offsets())
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    err = plan.device_error()
    assert err & B.MP_ERR_TIMEOUT, err
    assert err & B.MP_ERR_INVALID_ARG, err
    assert elapsed < 30.0
    # the context is still usable: re-zero the workspace and run the real thing
    plan.workspace.zero_()
    plan.dev_err.zero_()
    plan.step()
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    out, st = oracle.dispatch(wl.bf16_bits(inp.x), inp.topk_idx, inp.topk_weights, mask, inp.E)
    assert st == 0
    assert np.array_equal(plan.send_row.cpu().numpy(), out["send_row"])
    assert np.array_equal(wl.bf16_bits(plan.recv_x[:out["num_recv"]]), out["recv_x"])


@pytest.mark.parametrize("call", ["layout_and_offsets", "layout_dispatch"])
def test_grid_barrier_wait_times_out_and_context_survives(call):
    """The fused kernel's grid barrier: the arrival count it waits to reach is moved out
    of reach from the host (the barrier's base word preset to 2^30 above the count), so
    every block's bounded wait runs out and the call reports MP_ERR_TIMEOUT; a normal call
    on a re-zeroed workspace is then exact.  Through mp_layout_dispatch the row copy that
    follows the timed-out kernel still runs and stays inside its buffers."""
    inp = wl.make_ep(dict(R=4, N=2048, E=16, K=4, H=64, routing="uniform", dtype="bf16"), seed=2)
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H)
    plan.load(inp)
    torch.cuda.synchronize()
    plan.workspace[148:152].copy_(torch.tensor([0, 0, 0, 0x40], dtype=torch.uint8))  # 2^30
    plan.dev_err.zero_()
    t0 = time.time()
    B.check(getattr(plan, call)())
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert plan.device_error() & B.MP_ERR_TIMEOUT, plan.device_error()
    assert elapsed < 30.0
    plan.workspace.zero_()
    plan.dev_err.zero_()
    plan.step()
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ntpr, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    out, st = oracle.dispatch(wl.bf16_bits(inp.x), inp.topk_idx, inp.topk_weights, mask, inp.E)
    assert st == 0
    assert np.array_equal(plan.num_tokens_per_rank.cpu().numpy(), ntpr)
    assert np.array_equal(plan.send_row.cpu().numpy(), out["send_row"])
    assert np.array_equal(wl.bf16_bits(plan.recv_x[:out["num_recv"]]), out["recv_x"])
