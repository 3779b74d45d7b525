"""mp_dispatch_noalloc against mp_dispatch.

mp_dispatch_noalloc serves callers that cannot allocate device memory for a
workspace (an application that reserves nearly all device memory for its own
pool, a plugin whose host framework owns every allocation, or a loop in which
cudaMalloc would synchronise the device).  It keeps the scan's scratch in a
fixed array inside the library instead.  These tests call it through the C
ABI and check that two calls in a row give exactly what the workspace-taking
mp_dispatch gives (dispatch outputs are indices and copied bytes, so the bar
is bit-exact), and that a problem too large for the fixed array is refused.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test; it also passes on its own.
"""
import numpy as np
import pytest
import torch

from combine_mp_layout_gb300 import binding as B
from combine_mp_layout_gb300 import workloads as wl
from combine_mp_layout_gb300.pipeline import EPPlan

pytestmark = pytest.mark.gpu

OUTPUTS = ("recv_x", "recv_src_rank", "recv_src_idx", "recv_topk_idx", "recv_topk_weights",
           "dest_offsets", "rank_prefix", "num_recv_tokens_per_expert", "send_row")


def _noalloc(plan: EPPlan, out: dict) -> int:
    return B.mp_dispatch_noalloc(
        plan.R, plan.N, plan.K, plan.E, plan.H, B.MP_BF16, plan.x, None, plan.topk_idx,
        plan.topk_weights, plan.is_token_in_rank, plan.num_tokens_per_rank,
        plan.num_tokens_per_expert, plan.cap, out["recv_x"], None, out["recv_src_rank"],
        out["recv_src_idx"], out["recv_topk_idx"], out["recv_topk_weights"],
        out["dest_offsets"], out["rank_prefix"], out["num_recv_tokens_per_expert"],
        out["send_row"], out["dev_err"])


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy() if t.element_size() == 1 else (
        t.view(torch.int16).numpy() if t.element_size() == 2 else t.view(torch.int32).numpy())


def test_noalloc_matches_dispatch_on_two_calls_in_a_row():
    plan = EPPlan(8, 1000, 8, 256, 256, "bf16")
    out = {k: torch.full_like(getattr(plan, k), -3) if k != "recv_x" else
           torch.zeros_like(plan.recv_x) for k in OUTPUTS}
    out["dev_err"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((21, 22)):  # two calls in a row, different routing
        plan.load(wl.make_ep("dsv3", seed=seed, N=1000, H=256))
        plan.dev_err.zero_()
        B.check(plan.layout(), "mp_layout")
        B.check(plan.dispatch(), "mp_dispatch")
        B.check(_noalloc(plan, out), "mp_dispatch_noalloc")
        torch.cuda.synchronize()
        assert plan.device_error() == 0 and int(out["dev_err"].item()) == 0
        T = plan.num_recv()
        assert T > 0
        for k in OUTPUTS:
            want = getattr(plan, k)
            got = out[k]
            if k.startswith("recv_"):
                want, got = want[:T], got[:T]
            assert np.array_equal(_bits(got), _bits(want)), "call %d: %s differs" % (call, k)


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # mp_workspace_size(32, 100000, 256) is above the fixed 1 MiB; the call must be
    # refused before anything is launched (all pointers NULL, so nothing could run).
    assert B.mp_workspace_size(32, 100000, 256) > (1 << 20)
    f = B.lib().mp_dispatch_noalloc
    import ctypes
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i64,
                  P, P, P, P, P, P, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    st = f(32, 100000, 8, 256, 7168, B.MP_BF16, *([None] * 7), 10, *([None] * 12))
    assert st == B.MP_ERR_INVALID_ARG
