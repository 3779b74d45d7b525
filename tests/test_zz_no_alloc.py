"""mp_dispatch_noalloc against mp_dispatch.

mp_dispatch_noalloc serves callers that cannot allocate device memory for a
workspace (an application that reserves nearly all device memory for its own
pool, a plugin whose host framework owns every allocation, or a loop in which
cudaMalloc would synchronise the device).  It keeps the scan's scratch in a
fixed array inside the library instead.  These tests call it through the C
ABI and check that two calls in a row give exactly what the workspace-taking
mp_dispatch gives (dispatch outputs are indices and copied bytes, so the bar
is bit-exact), and that a problem too large for the fixed array is refused.
One test runs in a fresh process whose first calls are made on a
non-blocking stream, where the one-time zero-fill of the array must still be
complete before any call uses it.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test; it also passes on its own.
"""
import os
import subprocess
import sys

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


_FRESH_PROCESS = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, %(root)r)
from combine_mp_layout_gb300 import binding as B
from combine_mp_layout_gb300 import workloads as wl
from combine_mp_layout_gb300.pipeline import EPPlan

OUTPUTS = %(outputs)r
plan = EPPlan(8, 700, 8, 256, 128, "bf16")
out = {k: torch.full_like(getattr(plan, k), -3) for k in OUTPUTS}
out["dev_err"] = torch.zeros(1, dtype=torch.int32, device="cuda")

def noalloc(dev_err):
    return B.mp_dispatch_noalloc(
        plan.R, plan.N, plan.K, plan.E, plan.H, B.MP_BF16, plan.x, None, plan.topk_idx,
        plan.topk_weights, plan.is_token_in_rank, plan.num_tokens_per_rank,
        plan.num_tokens_per_expert, plan.cap, out["recv_x"], None, out["recv_src_rank"],
        out["recv_src_idx"], out["recv_topk_idx"], out["recv_topk_weights"],
        out["dest_offsets"], out["rank_prefix"], out["num_recv_tokens_per_expert"],
        out["send_row"], dev_err)

side = torch.cuda.Stream()  # torch's pool streams do not synchronise with the legacy stream
for call, seed in enumerate((41, 42)):
    plan.load(wl.make_ep("dsv3", seed=seed, N=700, H=128))
    plan.dev_err.zero_()
    B.check(plan.layout(), "mp_layout")
    B.check(plan.dispatch(), "mp_dispatch")
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        if call == 0:  # the process's first call is refused (no error word) and sets nothing up
            assert noalloc(None) == B.MP_ERR_INVALID_ARG
        B.check(noalloc(out["dev_err"]), "mp_dispatch_noalloc")
    torch.cuda.synchronize()
    assert plan.device_error() == 0 and int(out["dev_err"].item()) == 0
    T = plan.num_recv()
    for k in OUTPUTS:
        want, got = getattr(plan, k), out[k]
        if k.startswith("recv_"):
            want, got = want[:T], got[:T]
        a = got.detach().cpu().contiguous().view(torch.uint8).numpy()
        b = want.detach().cpu().contiguous().view(torch.uint8).numpy()
        assert np.array_equal(a, b), "call %%d: %%s differs" %% (call, k)
print("fresh-process noalloc ok")
"""


def test_noalloc_first_calls_on_a_non_blocking_stream_in_a_fresh_process():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = _FRESH_PROCESS % {"root": root, "outputs": OUTPUTS}
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "fresh-process noalloc ok" in r.stdout
