"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: bit-exact for counts, masks, offsets, send_row, receive metadata and
copied payload bytes (bf16 and e4m3); combine / reduce-scatterv within
1 bf16 ulp of the oracle's fp32 ascending-order sum rounded once (both sides
use the same order and rounding, so 0 ulp is what is expected; the bar is
the stated tolerance).  Sizes span several scan tiles / layout blocks with
ragged tails, ragged hidden sizes, R from 1 to 32, masked entries, empty
inputs, capacity overflow and bad expert ids; the full-size workloads run
in the launch configuration the benchmark times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_mp_layout_gb300 import binding as B
from combine_mp_layout_gb300 import workloads as wl
from combine_mp_layout_gb300.pipeline import EPPlan, RSVPlan
from tests import pins

pytestmark = pytest.mark.gpu

ULP_TOL = 1  # combine / reduce-scatterv: at most 1 bf16 ulp from the oracle


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns (ordered-integer map)."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7fff), 0x8000 + b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


# the largest distance seen by each check, reported at the end of the run
MAX_ULP_SEEN: dict = {}


def assert_bf16_close(got_bits, want_bits, what):
    """The contract bar (at most ULP_TOL bf16 ulp from the oracle), then exactness:
    both sides add in the same order and round once, so any non-zero distance is a
    regression even where the bar still holds."""
    d = ulp_distance(np.asarray(got_bits), np.asarray(want_bits))
    worst = int(d.max()) if d.size else 0
    MAX_ULP_SEEN[what] = max(worst, MAX_ULP_SEEN.get(what, 0))
    assert worst <= ULP_TOL, "%s: max %d ulp at %r" % (
        what, worst, np.unravel_index(int(d.argmax()), d.shape))
    assert worst == 0, "%s: within the bar but not bit-exact (max %d ulp)" % (what, worst)


def run_gpu(inp: wl.EPInputs, recv_capacity=None, y: torch.Tensor | None = None,
            repeat: int = 1) -> EPPlan:
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H, inp.dtype, recv_capacity)
    plan.load(inp)
    for _ in range(repeat):
        plan.dev_err.zero_()
        B.check(plan.layout(), "mp_layout")
        B.check(plan.dispatch(), "mp_dispatch")
        B.check(plan.combine(y), "mp_combine")
    torch.cuda.synchronize()
    return plan


def x_host(inp: wl.EPInputs) -> np.ndarray:
    return wl.bf16_bits(inp.x) if inp.dtype == "bf16" else wl.u8_bits(inp.x)


def compare_ep(inp: wl.EPInputs, plan: EPPlan, recv_capacity=None, y_bits=None,
               expect_err: int = 0, what: str = "combine"):
    R, N, E = inp.R, inp.N, inp.E
    ntpr, ntpe, mask, st = oracle.layout(inp.topk_idx, E)
    xs = inp.x_scales.numpy() if inp.x_scales is not None else None
    out, st2 = oracle.dispatch(x_host(inp), inp.topk_idx, inp.topk_weights, mask, E,
                               x_scales=xs, recv_capacity=recv_capacity)
    assert (st | st2) == expect_err == plan.device_error(), (st, st2, plan.device_error())
    assert np.array_equal(plan.num_tokens_per_rank.cpu().numpy(), ntpr)
    assert np.array_equal(plan.num_tokens_per_expert.cpu().numpy(), ntpe)
    assert np.array_equal(plan.is_token_in_rank.cpu().numpy().view(np.uint32), mask)
    for key in ("dest_offsets", "rank_prefix", "num_recv_tokens_per_expert", "send_row"):
        assert np.array_equal(getattr(plan, key).cpu().numpy(), out[key]), key
    n = min(out["num_recv"], plan.cap)
    assert np.array_equal(plan.recv_src_rank[:n].cpu().numpy(), out["recv_src_rank"])
    assert np.array_equal(plan.recv_src_idx[:n].cpu().numpy(), out["recv_src_idx"])
    assert np.array_equal(plan.recv_topk_idx[:n].cpu().numpy(), out["recv_topk_idx"])
    assert np.array_equal(plan.recv_topk_weights[:n].cpu().numpy().view(np.uint32),
                          out["recv_topk_weights"].view(np.uint32))
    got_x = wl.bf16_bits(plan.recv_x[:n]) if inp.dtype == "bf16" else wl.u8_bits(plan.recv_x[:n])
    assert np.array_equal(got_x, out["recv_x"]), "recv_x bytes"
    if xs is not None:
        assert np.array_equal(plan.recv_scales[:n].cpu().numpy().view(np.uint32),
                              out["recv_scales"].view(np.uint32))
    if inp.dtype == "bf16" or y_bits is not None:
        yb = out["recv_x"] if y_bits is None else y_bits
        comb, st3 = oracle.combine(yb, out["send_row"])
        assert st3 == 0
        assert_bf16_close(wl.bf16_bits(plan.out), comb, what)
    return out


def run_gpu_fused(inp: wl.EPInputs, recv_capacity=None, y: torch.Tensor | None = None,
                  repeat: int = 1) -> EPPlan:
    """As run_gpu, with mp_layout_and_offsets in place of mp_layout + mp_dispatch_offsets."""
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H, inp.dtype, recv_capacity)
    plan.load(inp)
    for _ in range(repeat):
        plan.dev_err.zero_()
        B.check(plan.layout_and_offsets(), "mp_layout_and_offsets")
        B.check(plan.dispatch_rows(), "mp_dispatch_rows")
        B.check(plan.combine(y), "mp_combine")
    torch.cuda.synchronize()
    return plan


# ---------------------------------------------------------------------------
# small and fuzzed shapes
# ---------------------------------------------------------------------------
def test_tiny_config():
    inp = wl.make_ep("tiny", seed=0)
    compare_ep(inp, run_gpu(inp))


def test_hand_fixture_on_gpu():
    g = pins.load("ep_hand_r2.json")
    ex = g["expect"]
    R, N, E, K = g["R"], g["N"], g["E"], g["K"]
    x = torch.zeros((R, N, 8), dtype=torch.float32)
    x[..., :2] = torch.tensor(g["x"])
    inp = wl.EPInputs(R, N, 8, E, K, "bf16", np.array(g["topk_idx"], np.int32),
                      np.array(g["topk_weights"], np.float32), x.to(torch.bfloat16))
    plan = run_gpu(inp)
    assert plan.num_tokens_per_rank.cpu().tolist() == ex["num_tokens_per_rank"]
    assert plan.num_tokens_per_expert.cpu().tolist() == ex["num_tokens_per_expert"]
    assert plan.is_token_in_rank.cpu().tolist() == ex["is_token_in_rank"]
    for key in ("dest_offsets", "rank_prefix", "num_recv_tokens_per_expert", "send_row"):
        assert getattr(plan, key).cpu().tolist() == ex[key], key
    T = ex["dest_offsets"][-1]
    assert plan.recv_src_rank[:T].cpu().tolist() == ex["recv_src_rank"]
    assert plan.recv_src_idx[:T].cpu().tolist() == ex["recv_src_idx"]
    assert plan.recv_topk_idx[:T].cpu().tolist() == ex["recv_topk_idx"]
    assert plan.recv_topk_weights[:T].cpu().tolist() == ex["recv_topk_weights"]
    assert plan.recv_x[:T, :2].float().cpu().tolist() == ex["recv_x"]
    assert plan.out[..., :2].float().cpu().tolist() == ex["combine_of_recv_x"]
    y = torch.zeros((T, 8), dtype=torch.bfloat16, device="cuda")
    y[:, :2] = torch.tensor(ex["y"], dtype=torch.bfloat16)
    B.check(plan.combine(y))
    torch.cuda.synchronize()
    assert plan.out[..., :2].float().cpu().tolist() == ex["combine_of_y"]


def test_sum_order_fixture_on_gpu():
    g = pins.load("sum_order_r3.json")
    rows = torch.tensor(g["rows_in_rank_order"], dtype=torch.float32).to(torch.bfloat16).cuda()
    want = [int(h, 16) for h in g["expect_bf16_bits"]]
    send_row = torch.full((3, 1, 3), -1, dtype=torch.int32, device="cuda")
    send_row[0, 0] = torch.tensor([0, 1, 2], dtype=torch.int32)
    out = torch.full((3, 1, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.check(B.mp_combine(3, 1, 8, rows, 3, send_row, out, err))
    rs_out = torch.full((1, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    B.check(B.mp_reducescatterv(3, 8, [0, 1, 0], rows.reshape(3, 1, 8).contiguous(), rs_out))
    torch.cuda.synchronize()
    assert wl.bf16_bits(out[0, 0]).tolist() == want
    assert not wl.bf16_bits(out[1:]).any()
    assert wl.bf16_bits(rs_out[0]).tolist() == want
    assert int(err.item()) == 0


def assert_bits_or_both_nan(got_bits, want_bits, what):
    """Bit-exact where the oracle's result is a number (infinities included); a NaN
    where it is a NaN (NaN payloads are not compared)."""
    g = np.asarray(got_bits).astype(np.uint32)
    w = np.asarray(want_bits).astype(np.uint32)
    gn = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    wn = ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
    assert np.array_equal(gn, wn), "%s: NaN positions differ (%d vs %d)" % (
        what, int(gn.sum()), int(wn.sum()))
    bad = np.nonzero(g[~wn] != w[~wn])[0]
    assert bad.size == 0, "%s: %d results differ, first %s vs %s" % (
        what, bad.size, hex(int(g[~wn][bad[0]])), hex(int(w[~wn][bad[0]])))


def _tb(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def test_nonfinite_sums_match_oracle():
    """Infinities, NaNs, signed zeros and sums past bf16's or binary32's largest value,
    through the combine and the reduce-scatterv: the IEEE closed forms the oracle is
    pinned to, then random rows with such values sprinkled in."""
    H = 8
    for addends, _ in pins.NONFINITE_CASES:
        n = len(addends)
        rows = pins._bits(np.repeat(np.array(addends, np.float32)[:, None], H, axis=1))
        send_row = np.full((n, 1, n), -1, np.int32)
        send_row[0, 0] = np.arange(n)
        want, st = oracle.combine(rows, send_row)
        out = torch.zeros((n, 1, H), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.check(B.mp_combine(n, 1, H, _tb(rows), n, torch.from_numpy(send_row).cuda(), out, err))
        sizes = [0] * n
        sizes[n - 1] = 1
        want_rs, st2 = oracle.reducescatterv(rows.reshape(n, 1, H), sizes)
        rs = torch.zeros((1, H), dtype=torch.bfloat16, device="cuda")
        B.check(B.mp_reducescatterv(n, H, sizes, _tb(rows.reshape(n, 1, H)), rs))
        torch.cuda.synchronize()
        assert st == st2 == 0 and int(err.item()) == 0
        assert_bits_or_both_nan(wl.bf16_bits(out), want, "combine %r" % (addends,))
        assert_bits_or_both_nan(wl.bf16_bits(rs), want_rs, "reduce-scatterv %r" % (addends,))
    # random rows, 1% each of +Inf, -Inf, NaN, +-bf16 max and -0.0 among N(0,1) values
    inp = wl.make_ep(dict(R=4, N=300, E=16, K=4, H=136, routing="uniform", dtype="bf16"), seed=77)
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H)
    plan.load(inp)
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    torch.cuda.synchronize()
    rng = np.random.default_rng(78)

    def sprinkle(shape):
        v = rng.standard_normal(shape).astype(np.float32)
        u = rng.random(shape)
        special = [np.inf, -np.inf, np.nan, 3.3895314e38, -3.3895314e38, -0.0]
        for i, val in enumerate(special):
            v[(u >= i * 0.01) & (u < (i + 1) * 0.01)] = val
        return pins._bits(v)

    y = sprinkle((plan.cap, inp.H))
    B.check(plan.combine(_tb(y)))
    torch.cuda.synchronize()
    want, st = oracle.combine(y, plan.send_row.cpu().numpy())
    assert st == 0 and plan.device_error() == 0
    assert_bits_or_both_nan(wl.bf16_bits(plan.out), want, "combine, sprinkled")
    sizes = [7, 0, 130, 1, 64]
    x = sprinkle((5, sum(sizes), 136))
    rs = torch.zeros((sum(sizes), 136), dtype=torch.bfloat16, device="cuda")
    B.check(B.mp_reducescatterv(5, 136, sizes, _tb(x), rs))
    torch.cuda.synchronize()
    want_rs, st = oracle.reducescatterv(x, sizes)
    assert st == 0
    assert_bits_or_both_nan(wl.bf16_bits(rs), want_rs, "reduce-scatterv, sprinkled")
    # the weighted low-latency combine: products and sums in binary32 (0 * Inf = NaN)
    ll, st = oracle.dispatch_ll(np.zeros((inp.R, inp.N, 8), np.uint16), inp.topk_idx, inp.E)
    assert st == 0
    yl = sprinkle((ll["num_recv"], 136))
    w = inp.topk_weights.copy()
    w[:, ::9, 0] = 0.0
    want_ll, st = oracle.combine_ll(yl, ll["slot_row"], w)
    out = torch.zeros((inp.R, inp.N, 136), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.check(B.mp_combine_ll(inp.R, inp.N, inp.K, 136, _tb(yl), ll["num_recv"],
                            torch.from_numpy(ll["slot_row"]).cuda(), torch.from_numpy(w).cuda(),
                            out, err))
    torch.cuda.synchronize()
    assert st == 0 and int(err.item()) == 0
    assert_bits_or_both_nan(wl.bf16_bits(out), want_ll, "weighted LL combine, sprinkled")


def test_weighted_combine_closed_forms_on_gpu():
    """The weighted LL combine on the closed forms its oracle is pinned to: the
    sum-order fixture with unit weights (slots in ascending k, a masked slot skipped),
    and a product rounded before it is added (w = 1 + 2^-20, y = 1 + 2^-7, then -w:
    +0, not the -2^-27 a fused multiply-add would leave)."""
    g = pins.load("sum_order_r3.json")
    rows = pins._bits(g["rows_in_rank_order"])
    want = [int(h, 16) for h in g["expect_bf16_bits"]]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for slots in ([0, 1, 2], [0, -1, 1, 2]):
        k = len(slots)
        out = torch.full((1, 1, 8), 7.0, dtype=torch.bfloat16, device="cuda")
        B.check(B.mp_combine_ll(1, 1, k, 8, _tb(rows), 3,
                                torch.tensor([[slots]], dtype=torch.int32, device="cuda"),
                                torch.ones((1, 1, k), dtype=torch.float32, device="cuda"), out, err))
        torch.cuda.synchronize()
        assert wl.bf16_bits(out[0, 0]).tolist() == want, slots
    y = pins._bits(np.full((2, 8), 1.0 + 2.0**-7, np.float32))
    w = torch.tensor([[[1.0 + 2.0**-20, -(1.0 + 2.0**-20)]]], dtype=torch.float32, device="cuda")
    out = torch.full((1, 1, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    B.check(B.mp_combine_ll(1, 1, 2, 8, _tb(y), 2,
                            torch.tensor([[[0, 1]]], dtype=torch.int32, device="cuda"), w, out,
                            err))
    torch.cuda.synchronize()
    assert not wl.bf16_bits(out).any(), wl.bf16_bits(out)
    assert int(err.item()) == 0


FUZZ = [  # R, N, E, K, H  (N not a multiple of 256, H not a multiple of a slab)
    (1, 100, 4, 2, 64),
    (2, 257, 8, 2, 136),
    (3, 300, 12, 3, 264),
    (4, 513, 16, 4, 8),
    (5, 257, 20, 6, 1032),
    (8, 1000, 64, 8, 520),
    (16, 130, 32, 3, 96),
    (32, 40, 64, 8, 16),
    (7, 777, 28, 28, 24),   # K = E: every token to every rank
    (2, 9000, 8, 3, 16),    # more than 8192 tokens per rank: multi-block layout
    (4, 300, 64, 32, 16),   # the largest top-k
    (32, 50, 64, 32, 16),   # the largest rank count and top-k: 49 KB of scan staging
    (2, 40, 8, 2, 32776),   # 64 KB rows, 16-byte vectors
    (3, 30, 6, 2, 30720),   # 60 KB rows, 32-byte vectors
]


@pytest.mark.parametrize("shape", FUZZ, ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s)
def test_fuzz_shapes(shape):
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"),
                     seed=R * 1000 + N)
    if K < E:  # mask some entries and a few whole tokens
        rng = np.random.default_rng(N)
        idx = inp.topk_idx.copy()
        idx[rng.random(idx.shape) < 0.1] = -1
        idx[:, ::17, :] = -1
        inp.topk_idx = idx
    y = wl.random_bf16((R * N * min(R, K), H), seed=N)
    plan = run_gpu(inp, y=y.cuda())
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y))


def test_zipf_small():
    inp = wl.make_ep("skew", seed=3, N=300, H=64)
    compare_ep(inp, run_gpu(inp))


def test_fp8_small():
    inp = wl.make_ep("fp8", seed=4, N=333, H=384)
    y = wl.random_bf16((inp.R * inp.N * 8, inp.H), seed=4)
    plan = run_gpu(inp, y=y.cuda())
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y))


def test_repeated_calls_reuse_workspace():
    """The scan's tile states are tagged per launch: back-to-back calls on one
    workspace (and a changed routing in between) stay exact."""
    inp = wl.make_ep("dsv3", seed=6, N=700, H=64)
    plan = run_gpu(inp, repeat=3)
    compare_ep(inp, plan)
    inp2 = wl.make_ep("dsv3", seed=7, N=700, H=64)
    plan.load(inp2)
    for _ in range(2):
        plan.dev_err.zero_()
        plan.step()
    torch.cuda.synchronize()
    compare_ep(inp2, plan)


def test_split_dispatch_and_cached_rows():
    """mp_dispatch_offsets + mp_dispatch_rows equal mp_dispatch, and one set of offsets
    dispatches a second payload routed the same way (e4m3 with scales too)."""
    for dtype, H in (("bf16", 264), ("e4m3", 256)):
        inp = wl.make_ep(dict(R=6, N=500, E=24, K=4, H=H, routing="uniform", dtype=dtype), seed=9)
        plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H, dtype)
        plan.load(inp)
        B.check(plan.layout())
        B.check(plan.dispatch_offsets())
        B.check(plan.dispatch_rows())
        B.check(plan.combine(wl.random_bf16((plan.cap, H), 1).cuda()) if dtype != "bf16"
                else plan.combine())
        torch.cuda.synchronize()
        compare_ep(inp, plan, y_bits=wl.bf16_bits(wl.random_bf16((plan.cap, H), 1))
                   if dtype != "bf16" else None)
        # a second payload, same routing: only the row copy runs
        inp2 = wl.make_ep(dict(R=6, N=500, E=24, K=4, H=H, routing="uniform", dtype=dtype),
                          seed=9)
        g = torch.Generator().manual_seed(123)
        x2 = torch.randn((inp.R, inp.N, H), generator=g)
        inp2.x = x2.to(torch.bfloat16) if dtype == "bf16" else x2.to(torch.float8_e4m3fn)
        if dtype != "bf16":
            inp2.x_scales = torch.rand((inp.R, inp.N, H // 128), generator=g) + 0.5
        recv2 = torch.zeros_like(plan.recv_x)
        rs2 = torch.zeros_like(plan.recv_scales) if dtype != "bf16" else None
        B.check(plan.dispatch_rows(x=inp2.x.cuda(),
                                   x_scales=inp2.x_scales.cuda() if dtype != "bf16" else None,
                                   recv_x=recv2, recv_scales=rs2))
        torch.cuda.synchronize()
        _, _, mask, _ = oracle.layout(inp2.topk_idx, inp2.E)
        xs = inp2.x_scales.numpy() if dtype != "bf16" else None
        out, st = oracle.dispatch(x_host(inp2), inp2.topk_idx, inp2.topk_weights, mask, inp2.E,
                                  x_scales=xs)
        n = out["num_recv"]
        got = wl.bf16_bits(recv2[:n]) if dtype == "bf16" else wl.u8_bits(recv2[:n])
        assert st == 0 and np.array_equal(got, out["recv_x"])
        if xs is not None:
            assert np.array_equal(rs2[:n].cpu().numpy().view(np.uint32),
                                  out["recv_scales"].view(np.uint32))


@pytest.mark.parametrize("shape", [(4, 300, 16, 4, 384), (3, 129, 12, 2, 128),
                                   (8, 4096, 256, 8, 7168)],
                         ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s)
def test_dispatch_rows_e4m3_quantises_like_the_oracle(shape):
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=H)
    x = inp.x.float()
    x[0, 0, :128] = 0.0                      # an all-zero block
    x[0, 1, :] = 3.0                         # constant blocks
    x[R - 1, N - 1, -128:] *= 1e-3           # a block of small values (subnormal codes)
    inp.x = x.to(torch.bfloat16)
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    rq = torch.zeros((plan.cap, H), dtype=torch.uint8, device="cuda")
    rs = torch.zeros((plan.cap, H // 128), dtype=torch.float32, device="cuda")
    B.check(B.mp_dispatch_rows_e4m3(R, N, H, plan.x, plan.send_row, plan.cap, rq, rs))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    q, sc, st = oracle.quantize_e4m3(wl.bf16_bits(inp.x))
    _, _, mask, _ = oracle.layout(inp.topk_idx, E)
    out, st2 = oracle.dispatch(q, inp.topk_idx, inp.topk_weights, mask, E, x_scales=sc)
    assert st == st2 == 0
    n = out["num_recv"]
    assert np.array_equal(rq[:n].cpu().numpy(), out["recv_x"])
    assert np.array_equal(rs[:n].cpu().numpy().view(np.uint32), out["recv_scales"].view(np.uint32))


@pytest.mark.parametrize("shape", [(4, 300, 16, 4, 96), (8, 4096, 256, 8, 7168)],
                         ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s)
def test_dispatch_rows_mxfp8_quantises_like_the_oracle(shape):
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=H + 1)
    x = inp.x.float()
    x[0, 0, :32] = 0.0                          # all-zero block: code 0
    x[0, 1, 32:64] = 2.0**-130                  # tiny non-zero block: code 0, kept
    x[R - 1, 2, :] *= 300.0                     # large values: saturation above 448 * X
    x[1, 3, :32] *= torch.exp2(torch.arange(32, dtype=torch.float32) - 16)  # wide range
    inp.x = x.to(torch.bfloat16)
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    rq = torch.zeros((plan.cap, H), dtype=torch.uint8, device="cuda")
    rc = torch.zeros((plan.cap, H // 32), dtype=torch.uint8, device="cuda")
    B.check(B.mp_dispatch_rows_mxfp8(R, N, H, plan.x, plan.send_row, plan.cap, rq, rc))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    q, codes, st = oracle.quantize_mxfp8(wl.bf16_bits(inp.x))
    assert st == 0
    payload = np.concatenate([q, codes], axis=-1)  # dispatch codes and elements as one byte row
    _, _, mask, _ = oracle.layout(inp.topk_idx, E)
    out, st2 = oracle.dispatch(payload, inp.topk_idx, inp.topk_weights, mask, E)
    assert st2 == 0
    n = out["num_recv"]
    assert np.array_equal(rq[:n].cpu().numpy(), out["recv_x"][:, :H])
    assert np.array_equal(rc[:n].cpu().numpy(), out["recv_x"][:, H:])


@pytest.mark.parametrize("shape", [(4, 300, 16, 4, 96), (8, 4096, 256, 8, 7168)],
                         ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s)
def test_dispatch_rows_mxfp4_quantises_like_the_oracle(shape):
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=H + 2)
    inp.x = _special_blocks(inp.x.reshape(R * N, H), 32).reshape(R, N, H)
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    rq = torch.zeros((plan.cap, H // 2), dtype=torch.uint8, device="cuda")
    rc = torch.zeros((plan.cap, H // 32), dtype=torch.uint8, device="cuda")
    B.check(B.mp_dispatch_rows_mxfp4(R, N, H, plan.x, plan.send_row, plan.cap, rq, rc))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    q, codes = _oracle_quant("mxfp4", inp.x)
    payload = np.concatenate([q, codes], axis=-1)
    _, _, mask, _ = oracle.layout(inp.topk_idx, E)
    out, st2 = oracle.dispatch(payload, inp.topk_idx, inp.topk_weights, mask, E)
    assert st2 == 0
    n = out["num_recv"]
    assert np.array_equal(rq[:n].cpu().numpy(), out["recv_x"][:, :H // 2])
    assert np.array_equal(rc[:n].cpu().numpy(), out["recv_x"][:, H // 2:])


@pytest.mark.parametrize("dtype,shape,cap_frac", [
    ("bf16", (4, 300, 16, 4, 384), None), ("e4m3", (3, 129, 12, 2, 256), None),
    ("bf16", (5, 77, 20, 3, 8200), None), ("bf16", (4, 300, 16, 4, 64), 0.5),
    ("bf16", (8, 4096, 256, 8, 7168), None)],
    ids=["bf16", "e4m3_scales", "rows_above_16KB", "capacity", "dsv3"])
def test_bulk_copy_dispatch_matches_the_oracle(dtype, shape, cap_frac):
    """mp_dispatch_rows_bulk (cp.async.bulk through shared memory) moves the same bytes
    as the oracle's dispatch, including rows cut into several 16 KB pieces."""
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype=dtype), seed=H)
    plan = EPPlan(R, N, K, E, H, dtype)
    plan.load(inp)
    B.check(plan.layout())
    cap = plan.cap
    if cap_frac is not None:
        torch.cuda.synchronize()
        cap = int(plan.num_tokens_per_rank.sum().item() * cap_frac)
    B.check(B.mp_dispatch_offsets(
        R, N, K, E, plan.topk_idx, plan.topk_weights, plan.is_token_in_rank,
        plan.num_tokens_per_rank, plan.num_tokens_per_expert, cap, plan.recv_src_rank,
        plan.recv_src_idx, plan.recv_topk_idx, plan.recv_topk_weights, plan.dest_offsets,
        plan.rank_prefix, plan.num_recv_tokens_per_expert, plan.send_row, plan.dev_err,
        plan.workspace))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.check(B.mp_dispatch_rows_bulk(R, N, H, B.MP_BF16 if dtype == "bf16" else B.MP_E4M3,
                                    plan.x, plan.x_scales, plan.send_row, cap, plan.recv_x,
                                    plan.recv_scales, err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _, _, mask, _ = oracle.layout(inp.topk_idx, E)
    xs = inp.x_scales.numpy() if dtype != "bf16" else None
    out, st = oracle.dispatch(x_host(inp), inp.topk_idx, inp.topk_weights, mask, E,
                              x_scales=xs, recv_capacity=cap)
    assert (st == 0) == (cap_frac is None)
    n = min(out["num_recv"], cap)
    got = wl.bf16_bits(plan.recv_x[:n]) if dtype == "bf16" else wl.u8_bits(plan.recv_x[:n])
    assert np.array_equal(got, out["recv_x"][:n])
    if xs is not None:
        assert np.array_equal(plan.recv_scales[:n].cpu().numpy().view(np.uint32),
                              out["recv_scales"][:n].view(np.uint32))


FUSED = [(1, 100, 4, 2, 64), (3, 300, 12, 3, 264), (8, 1000, 64, 8, 520), (16, 130, 32, 3, 96),
         (32, 40, 64, 8, 16), (7, 777, 28, 28, 24), (2, 9000, 8, 3, 16),
         (4, 257, 4, 2, 64),     # one expert per rank
         (3, 1, 6, 2, 64),       # a single token per rank
         (32, 300, 8192, 8, 16),  # the largest expert count: 32 KB of histogram per block
         (8, 64, 8192, 8, 64),    # few ids, but too many experts for the one-kernel form's tables
         (8, 20000, 32, 4, 16),  # more tiles than blocks, so blocks own several
         (32, 50, 64, 32, 16)]   # the largest rank count and top-k


@pytest.mark.parametrize("shape", FUSED, ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s)
def test_fused_layout_and_offsets(shape):
    """One cooperative launch for layout + offsets: the oracle's results, repeatedly
    (the workspace's barrier words, epochs and accumulators are reused)."""
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"),
                     seed=R * 1000 + N + 1)
    if K < E:
        idx = inp.topk_idx.copy()
        idx[np.random.default_rng(N).random(idx.shape) < 0.1] = -1
        idx[:, ::13, :] = -1
        inp.topk_idx = idx
    y = wl.random_bf16((R * N * min(R, K), H), seed=N + 1)
    plan = run_gpu_fused(inp, y=y.cuda(), repeat=3)
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y))


@pytest.mark.parametrize("name", ["dsv3", "skew"])
def test_fused_layout_and_offsets_full_size(name):
    """The benchmark's calls (fused layout + offsets, rows, combine) at full size, the
    combine fed fully random expert outputs so that its summation order is checked."""
    inp = wl.make_ep(name, seed=0)
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    rows = int(np.unpackbits(mask.view(np.uint8)).sum())
    y = wl.random_bf16_rows(rows, inp.H, seed=11)
    plan = run_gpu_fused(inp, y=y.cuda(), repeat=2)
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y), what="%s full-size step combine(y)" % name)


def run_gpu_one_call(inp: wl.EPInputs, recv_capacity=None, y: torch.Tensor | None = None,
                     repeat: int = 1) -> EPPlan:
    """As run_gpu, with the whole dispatch in one call (mp_layout_dispatch)."""
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H, inp.dtype, recv_capacity)
    plan.load(inp)
    for _ in range(repeat):
        plan.dev_err.zero_()
        B.check(plan.layout_dispatch(), "mp_layout_dispatch")
        B.check(plan.combine(y), "mp_combine")
    torch.cuda.synchronize()
    return plan


@pytest.mark.parametrize("shape", FUSED, ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s)
def test_one_call_dispatch(shape):
    """mp_layout_dispatch (one cooperative launch for layout + offsets, the row copy --
    which writes the receive metadata -- as its programmatic dependent): every output the
    oracle's layout -> dispatch gives, and the combine of random rows, call after call."""
    R, N, E, K, H = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"),
                     seed=R * 1000 + N + 2)
    if K < E:
        idx = inp.topk_idx.copy()
        idx[np.random.default_rng(N + 1).random(idx.shape) < 0.1] = -1
        idx[:, ::11, :] = -1
        inp.topk_idx = idx
    y = wl.random_bf16((R * N * min(R, K), H), seed=N + 2)
    plan = run_gpu_one_call(inp, y=y.cuda(), repeat=3)
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y), what="one-call step combine(y)")


@pytest.mark.parametrize("N", [128, 256, 512, 1024])
def test_one_call_dispatch_small_batches(N):
    """The DeepSeek-V3 shape at the small batches the benchmark also times (N tokens per
    rank): one-call dispatch (one kernel of 512-thread blocks at N=128, of 1,024-thread
    blocks at N=256, two launches above), then the combine of random rows."""
    inp = wl.make_ep("dsv3", seed=N, N=N)
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    rows = int(np.unpackbits(mask.view(np.uint8)).sum())
    y = wl.random_bf16_rows(rows, inp.H, seed=N)
    plan = run_gpu_one_call(inp, y=y.cuda(), repeat=2)
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y), what="dsv3 N=%d one-call combine(y)" % N)


@pytest.mark.parametrize("name", ["dsv3", "skew", "fp8"])
def test_one_call_dispatch_full_size(name):
    inp = wl.make_ep(name, seed=0)
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    rows = int(np.unpackbits(mask.view(np.uint8)).sum())
    y = wl.random_bf16_rows(rows, inp.H, seed=21)
    plan = run_gpu_one_call(inp, y=y.cuda(), repeat=2)
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y), what="%s full one-call combine(y)" % name)


def test_one_call_dispatch_e4m3_ragged():
    """e4m3 rows with their fp32 scales through the one-call dispatch, ragged tiles."""
    inp = wl.make_ep(dict(R=5, N=333, E=40, K=5, H=384, routing="uniform", dtype="e4m3"), seed=9)
    y = wl.random_bf16((inp.R * inp.N * 5, inp.H), seed=9)
    plan = run_gpu_one_call(inp, y=y.cuda(), repeat=2)
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y), what="e4m3 one-call combine(y)")


def test_one_call_dispatch_capacity_and_bad_ids():
    inp = wl.make_ep(dict(R=4, N=300, E=16, K=4, H=64, routing="uniform", dtype="bf16"), seed=4)
    inp.topk_idx[2, 5, 1] = 99
    inp.topk_idx[0, 7, 0] = -4
    plan = run_gpu_one_call(inp, recv_capacity=700)
    compare_ep(inp, plan, recv_capacity=700, expect_err=B.MP_ERR_CAPACITY | B.MP_ERR_BAD_EXPERT)


@pytest.mark.parametrize("cfg", [dict(R=5, N=77, E=20, K=6, H=2056, dtype="bf16"),
                                 dict(R=4, N=150, E=32, K=4, H=4096, dtype="e4m3"),
                                 dict(R=8, N=60, E=64, K=8, H=1024, dtype="bf16", cap=900),
                                 dict(R=2, N=3, E=8, K=2, H=20480, dtype="bf16"),
                                 dict(R=16, N=1, E=32, K=4, H=7168, dtype="bf16"),
                                 dict(R=4, N=256, E=16, K=4, H=16384, dtype="bf16"),
                                 dict(R=4, N=256, E=16, K=4, H=32768, dtype="e4m3"),
                                 dict(R=4, N=256, E=16, K=4, H=16384, dtype="bf16", cap=2000),
                                 dict(R=32, N=16, E=64, K=8, H=2048, dtype="bf16")],
                         ids=["ragged", "e4m3_scales", "capacity", "blocks_inside_a_token",
                              "one_token_per_rank", "large_part", "large_part_e4m3_scales",
                              "large_part_capacity", "32_ranks"])
def test_one_call_dispatch_bulk_copies(cfg):
    """mp_layout_dispatch at small batches with rows of 2 KB or more: one kernel whose
    blocks count every token, bulk-load their part of x and bulk-store each row piece.
    "large_part": 32 KB rows, so a block's part of x (over 192 KB) does not fit shared
    memory and the kernel copies through registers instead."""
    cfg = dict(cfg)
    cap = cfg.pop("cap", None)
    inp = wl.make_ep(dict(cfg, routing="uniform"), seed=cfg["N"] + cfg["H"])
    idx = inp.topk_idx.copy()
    idx[:, ::5, 0] = -1
    inp.topk_idx = idx
    y = wl.random_bf16((inp.R * inp.N * min(inp.R, inp.K), inp.H), seed=3)
    plan = run_gpu_one_call(inp, recv_capacity=cap, y=y.cuda(), repeat=2)
    compare_ep(inp, plan, recv_capacity=cap, y_bits=wl.bf16_bits(y),
               expect_err=B.MP_ERR_CAPACITY if cap is not None else 0,
               what="one-kernel dispatch combine(y)")


def test_one_call_dispatch_falls_back_beyond_one_grid():
    """Beyond one resident grid the one-call dispatch runs the layout, scan and row-copy
    kernels one after another, with the same results."""
    inp = wl.make_ep(dict(R=32, N=40000, E=64, K=2, H=8, routing="uniform", dtype="bf16"), seed=6)
    plan = run_gpu_one_call(inp)
    compare_ep(inp, plan)


def test_fused_layout_and_offsets_capacity_and_bad_ids():
    inp = wl.make_ep(dict(R=4, N=300, E=16, K=4, H=64, routing="uniform", dtype="bf16"), seed=4)
    inp.topk_idx[2, 5, 1] = 99
    plan = run_gpu_fused(inp, recv_capacity=700)
    compare_ep(inp, plan, recv_capacity=700, expect_err=B.MP_ERR_CAPACITY | B.MP_ERR_BAD_EXPERT)


@pytest.mark.parametrize("calls", ["one_call_dispatch", "three_calls"])
def test_step_replays_as_a_cuda_graph(calls):
    """The step captured in a CUDA graph and replayed: the oracle's results, replay after
    replay.  one_call_dispatch: mp_layout_dispatch (cooperative layout + offsets, then the
    row copy as its programmatic dependent) and the combine launched as the copy's
    dependent; three_calls: mp_layout_and_offsets, mp_dispatch_rows, mp_combine."""
    inp = wl.make_ep(dict(R=4, N=700, E=16, K=4, H=128, routing="uniform", dtype="bf16"), seed=8)
    plan = EPPlan(inp.R, inp.N, inp.K, inp.E, inp.H)
    plan.load(inp)
    step = plan.step if calls == "one_call_dispatch" else plan.step_three_calls
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # first calls (one-time launch setup) outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        for t in (plan.recv_src_rank, plan.recv_src_idx, plan.recv_topk_idx, plan.send_row):
            t.fill_(-7)
        plan.out.zero_()
        plan.recv_x.zero_()
        graph.replay()
    torch.cuda.synchronize()
    compare_ep(inp, plan)


def test_fused_layout_and_offsets_falls_back_beyond_one_grid():
    """R=32 x 40,000 tokens is 10,016 tiles, more than 16 per block of a resident grid:
    the call runs the two kernels instead, with the same results."""
    inp = wl.make_ep(dict(R=32, N=40000, E=64, K=2, H=8, routing="uniform", dtype="bf16"), seed=5)
    plan = run_gpu_fused(inp)
    compare_ep(inp, plan)


def test_empty_tokens():
    inp = wl.make_ep(dict(R=4, N=0, E=16, K=2, H=64, routing="uniform", dtype="bf16"))
    plan = run_gpu(inp)
    assert plan.num_tokens_per_rank.abs().sum().item() == 0
    assert plan.dest_offsets.abs().sum().item() == 0
    # the one-call layout + offsets and the whole step: every count and offset table is
    # written (zeros), whatever the buffers held before
    for t in (plan.num_tokens_per_rank, plan.num_tokens_per_expert, plan.dest_offsets,
              plan.rank_prefix, plan.num_recv_tokens_per_expert):
        t.fill_(-3)
    B.check(plan.layout_and_offsets())
    plan.step()
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    for t in (plan.num_tokens_per_rank, plan.num_tokens_per_expert, plan.dest_offsets,
              plan.rank_prefix, plan.num_recv_tokens_per_expert):
        assert not t.any().item()
        t.fill_(-3)
    plan.step_three_calls()
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    for t in (plan.num_tokens_per_rank, plan.num_tokens_per_expert, plan.dest_offsets,
              plan.rank_prefix, plan.num_recv_tokens_per_expert):
        assert not t.any().item()


def test_all_masked():
    inp = wl.make_ep(dict(R=3, N=50, E=6, K=2, H=64, routing="uniform", dtype="bf16"))
    inp.topk_idx[:] = -1
    plan = run_gpu(inp)
    compare_ep(inp, plan)
    assert not wl.bf16_bits(plan.out).any()


def test_capacity_overflow():
    inp = wl.make_ep(dict(R=4, N=300, E=16, K=4, H=64, routing="uniform", dtype="bf16"), seed=2)
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    total = int(np.unpackbits(mask.view(np.uint8)).sum())
    cap = total // 2
    plan = run_gpu(inp, recv_capacity=cap)
    compare_ep(inp, plan, recv_capacity=cap, expect_err=B.MP_ERR_CAPACITY)


def test_bad_expert_ids():
    inp = wl.make_ep(dict(R=2, N=64, E=8, K=2, H=64, routing="uniform", dtype="bf16"), seed=8)
    inp.topk_idx[0, 3, 0] = 8
    inp.topk_idx[1, 9, 1] = -5
    plan = run_gpu(inp)
    compare_ep(inp, plan, expect_err=B.MP_ERR_BAD_EXPERT)


def test_combine_rejects_rows_past_y():
    send_row = torch.tensor([[[0, 5]]], dtype=torch.int32, device="cuda").expand(2, 1, 2).contiguous()
    y = torch.ones((4, 8), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, 1, 8), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.check(B.mp_combine(2, 1, 8, y, 4, send_row, out, err))
    torch.cuda.synchronize()
    assert int(err.item()) & B.MP_ERR_CAPACITY
    assert out.float().cpu().eq(1.0).all()  # only row 0 was summed


@pytest.mark.parametrize("R,H,sizes", [(8, 64, [3, 0, 5, 1, 0, 2, 4, 1]), (3, 8, [0, 0, 0]),
                                       (5, 1032, [100, 0, 257, 3, 64]), (1, 72, [9])])
def test_rsv_agv_small(R, H, sizes):
    inp = wl.make_rsv(dict(R=R, H=H, sizes=sizes), seed=R + H)
    plan = RSVPlan(R, H, sizes)
    plan.x.copy_(inp.x)
    plan.shards.copy_(inp.shards)
    B.check(plan.reducescatterv())
    B.check(plan.allgatherv())
    torch.cuda.synchronize()
    rs, st = oracle.reducescatterv(wl.bf16_bits(inp.x), sizes)
    ag, st2 = oracle.allgatherv(wl.bf16_bits(inp.shards), sizes, R)
    assert st == st2 == 0
    assert_bf16_close(wl.bf16_bits(plan.rs_out), rs, "reducescatterv")
    assert np.array_equal(wl.bf16_bits(plan.ag_out), ag)


def test_global_ids_and_combined_weights():
    inp = wl.make_ep("skew", seed=12, N=700, H=64)
    R, N, K, E = inp.R, inp.N, inp.K, inp.E
    inp.topk_idx[:, ::9, 2] = -1
    plan = EPPlan(R, N, K, E, inp.H)
    plan.load(inp)
    B.check(plan.layout())
    gids = torch.full_like(plan.recv_topk_idx, -3)
    B.check(B.mp_dispatch_offsets_global(
        R, N, K, E, plan.topk_idx, plan.topk_weights, plan.is_token_in_rank,
        plan.num_tokens_per_rank, plan.num_tokens_per_expert, plan.cap, E, plan.recv_src_rank,
        plan.recv_src_idx, gids, plan.recv_topk_weights, plan.dest_offsets, plan.rank_prefix,
        plan.num_recv_tokens_per_expert, plan.send_row, plan.dev_err, plan.workspace))
    cw = torch.full((R, N, K), -3.0, device="cuda")
    B.check(B.mp_combine_weights(R, N, K, plan.recv_topk_weights, plan.cap, plan.send_row, cw,
                                 plan.dev_err))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    _, _, mask, _ = oracle.layout(inp.topk_idx, E)
    out, st = oracle.dispatch(np.zeros((R, N, 8), np.uint16), inp.topk_idx, inp.topk_weights,
                              mask, E)
    want_gid, st2 = oracle.recv_topk_global(inp.topk_idx, E, out, E)
    want_cw, st3 = oracle.combine_weights(out["recv_topk_weights"], out["send_row"])
    assert st == st2 == st3 == 0
    n = out["num_recv"]
    assert np.array_equal(gids[:n].cpu().numpy(), want_gid)
    assert np.array_equal(plan.send_row.cpu().numpy(), out["send_row"])
    assert np.array_equal(cw.cpu().numpy().view(np.uint32), want_cw.view(np.uint32))


@pytest.mark.parametrize("cfg", [dict(R=2, N=64, E=8, K=2, H=128), dict(R=8, N=128, E=256, K=8, H=7168),
                                 dict(R=5, N=77, E=20, K=6, H=264), dict(R=3, N=300, E=9, K=9, H=64),
                                 dict(R=4, N=3000, E=64, K=6, H=64),
                                 dict(R=8, N=64, E=8192, K=8, H=64),
                                 dict(R=4, N=500, E=16, K=4, H=64, cap_frac=0.5),
                                 dict(R=1, N=40, E=3, K=3, H=64)],
                         ids=lambda c: "R%(R)d_N%(N)d_E%(E)d_K%(K)d_H%(H)d" % c
                         + ("_cap" if "cap_frac" in c else ""))
@pytest.mark.parametrize("counts", ["layout", "self"])
def test_low_latency_layout_matches_oracle(cfg, counts):
    """counts: expert counts from mp_layout, or counted by the LL offsets call (NULL)."""
    cfg = dict(cfg)
    cap_frac = cfg.pop("cap_frac", None)
    inp = wl.make_ep(dict(cfg, routing="uniform", dtype="bf16"), seed=cfg["N"])
    R, N, E, K, H = cfg["R"], cfg["N"], cfg["E"], cfg["K"], cfg["H"]
    inp.topk_idx[:, ::7, 1] = -1
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    B.check(plan.layout())
    cap = R * N * K if cap_frac is None else int(R * N * K * cap_frac)
    dev = "cuda"
    eoff = torch.full((E + 1,), -3, dtype=torch.int32, device=dev)
    esoff = torch.full((E, R), -3, dtype=torch.int32, device=dev)
    src = torch.full((cap,), -3, dtype=torch.int32, device=dev)
    slot = torch.full((R, N, K), -3, dtype=torch.int32, device=dev)
    rx = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
    ntpe = plan.num_tokens_per_expert if counts == "layout" else None
    B.check(B.mp_dispatch_ll_offsets(R, N, K, E, plan.topk_idx, ntpe, cap,
                                     eoff, esoff, src, slot, plan.dev_err))
    B.check(B.mp_dispatch_ll_rows(R, N, K, H, B.MP_BF16, plan.x, None, slot, cap, rx, None))
    y = wl.random_bf16((cap, H), seed=N).cuda()
    out = torch.zeros((R, N, H), dtype=torch.bfloat16, device=dev)
    B.check(B.mp_combine_ll(R, N, K, H, y, cap, slot, plan.topk_weights, out, plan.dev_err))
    torch.cuda.synchronize()
    ll, st = oracle.dispatch_ll(wl.bf16_bits(inp.x), inp.topk_idx, E, recv_capacity=cap)
    assert plan.device_error() == st
    assert (st == 0) == (cap_frac is None)
    n = min(ll["num_recv"], cap)
    assert np.array_equal(eoff.cpu().numpy(), ll["expert_offsets"])
    assert np.array_equal(esoff.cpu().numpy(), ll["expert_src_offsets"])
    assert np.array_equal(slot.cpu().numpy(), ll["slot_row"])
    assert np.array_equal(src[:n].cpu().numpy(), ll["recv_src_token"])
    assert np.array_equal(wl.bf16_bits(rx[:n]), ll["recv_x"])
    comb, st = oracle.combine_ll(wl.bf16_bits(y), ll["slot_row"], inp.topk_weights)
    assert st == 0
    assert_bf16_close(wl.bf16_bits(out), comb, "combine_ll")


@pytest.mark.parametrize("cfg", [dict(R=2, N=64, E=8, K=2, H=128), dict(R=8, N=128, E=256, K=8, H=7168),
                                 dict(R=5, N=77, E=20, K=6, H=264), dict(R=4, N=3000, E=64, K=6, H=64),
                                 dict(R=32, N=40, E=64, K=4, H=64),
                                 dict(R=4, N=500, E=16, K=4, H=64, cap_frac=0.5),
                                 dict(R=1, N=40, E=3, K=3, H=64)],
                         ids=lambda c: "R%(R)d_N%(N)d_E%(E)d_K%(K)d_H%(H)d" % c
                         + ("_cap" if "cap_frac" in c else ""))
@pytest.mark.parametrize("counts", ["layout", "self"])
def test_low_latency_rank_major_matches_oracle(cfg, counts):
    cfg = dict(cfg)
    cap_frac = cfg.pop("cap_frac", None)
    inp = wl.make_ep(dict(cfg, routing="uniform", dtype="bf16"), seed=cfg["N"] + 1)
    R, N, E, K, H = cfg["R"], cfg["N"], cfg["E"], cfg["K"], cfg["H"]
    inp.topk_idx[:, ::5, 0] = -1
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    B.check(plan.layout())
    cap = R * N * K if cap_frac is None else int(R * N * K * cap_frac)
    dev = "cuda"
    doff = torch.full((R + 1,), -3, dtype=torch.int32, device=dev)
    dsoff = torch.full((R, R), -3, dtype=torch.int32, device=dev)
    src = torch.full((cap,), -3, dtype=torch.int32, device=dev)
    slot = torch.full((R, N, K), -3, dtype=torch.int32, device=dev)
    rx = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
    ntpe = plan.num_tokens_per_expert if counts == "layout" else None
    B.check(B.mp_dispatch_ll_offsets_rank_major(R, N, K, E, plan.topk_idx, ntpe, cap, doff, dsoff,
                                                src, slot, plan.dev_err))
    B.check(B.mp_dispatch_ll_rows(R, N, K, H, B.MP_BF16, plan.x, None, slot, cap, rx, None))
    y = wl.random_bf16((cap, H), seed=N + 1).cuda()
    out = torch.zeros((R, N, H), dtype=torch.bfloat16, device=dev)
    B.check(B.mp_combine_ll(R, N, K, H, y, cap, slot, plan.topk_weights, out, plan.dev_err))
    torch.cuda.synchronize()
    rm, st = oracle.dispatch_ll_rank_major(wl.bf16_bits(inp.x), inp.topk_idx, E, recv_capacity=cap)
    assert plan.device_error() == st
    assert (st == 0) == (cap_frac is None)
    n = min(rm["num_recv"], cap)
    assert np.array_equal(doff.cpu().numpy(), rm["dest_offsets"])
    assert np.array_equal(dsoff.cpu().numpy(), rm["dest_src_offsets"])
    assert np.array_equal(slot.cpu().numpy(), rm["slot_row"])
    assert np.array_equal(src[:n].cpu().numpy(), rm["recv_src_token"])
    assert np.array_equal(wl.bf16_bits(rx[:n]), rm["recv_x"])
    comb, st = oracle.combine_ll(wl.bf16_bits(y), rm["slot_row"], inp.topk_weights)
    assert st == 0
    assert_bf16_close(wl.bf16_bits(out), comb, "combine_ll rank-major")


def test_low_latency_rows_e4m3_with_scales():
    """The LL row copy of an e4m3 payload moves each row's scales with it."""
    R, N, E, K, H = 4, 200, 32, 4, 256
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="e4m3"), seed=31)
    plan = EPPlan(R, N, K, E, H, "e4m3")
    plan.load(inp)
    cap = R * N * K
    dev = "cuda"
    eoff = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    esoff = torch.zeros((E, R), dtype=torch.int32, device=dev)
    src = torch.zeros(cap, dtype=torch.int32, device=dev)
    slot = torch.zeros((R, N, K), dtype=torch.int32, device=dev)
    rx = torch.zeros((cap, H), dtype=torch.uint8, device=dev)
    rs = torch.zeros((cap, H // 128), dtype=torch.float32, device=dev)
    B.check(B.mp_dispatch_ll_offsets(R, N, K, E, plan.topk_idx, None, cap, eoff, esoff, src, slot,
                                     plan.dev_err))
    B.check(B.mp_dispatch_ll_rows(R, N, K, H, B.MP_E4M3, plan.x, plan.x_scales, slot, cap, rx, rs))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    payload = np.concatenate([wl.u8_bits(inp.x), inp.x_scales.numpy().view(np.uint8)], axis=-1)
    ll, st = oracle.dispatch_ll(payload, inp.topk_idx, E)
    assert st == 0
    n = ll["num_recv"]
    assert np.array_equal(slot.cpu().numpy(), ll["slot_row"])
    assert np.array_equal(rx[:n].cpu().numpy(), ll["recv_x"][:, :H])
    assert np.array_equal(rs[:n].cpu().numpy().view(np.uint8), ll["recv_x"][:, H:])


LL_ONE_CALL = [dict(R=2, N=64, E=8, K=2, H=128), dict(R=8, N=128, E=256, K=8, H=7168),
                 dict(R=5, N=77, E=20, K=6, H=264), dict(R=3, N=300, E=9, K=9, H=64),
                 dict(R=4, N=40, E=16, K=4, H=20480), dict(R=32, N=40, E=64, K=4, H=64),
                 dict(R=8, N=64, E=8192, K=8, H=64), dict(R=4, N=3000, E=64, K=6, H=64),
                 dict(R=4, N=500, E=16, K=4, H=64, cap_frac=0.5), dict(R=1, N=40, E=3, K=3, H=64),
                 dict(R=4, N=0, E=16, K=4, H=64), dict(R=2, N=50, E=64, K=32, H=64),
                 dict(R=16, N=1, E=32, K=4, H=64), dict(R=2, N=3, E=8, K=2, H=20480),
                 dict(R=4, N=100, E=2048, K=8, H=1024)]  # the one kernel's largest bin count


@pytest.mark.parametrize("cfg", LL_ONE_CALL, ids=lambda c: "R%(R)d_N%(N)d_E%(E)d_K%(K)d_H%(H)d" % c
                         + ("_cap" if "cap_frac" in c else ""))
@pytest.mark.parametrize("rank_major", [0, 1], ids=["expert_major", "rank_major"])
@pytest.mark.parametrize("counts", ["layout", "self"])
def test_low_latency_one_call_dispatch_matches_oracle(cfg, rank_major, counts):
    """mp_dispatch_ll against the oracle's LL layout and rows, three calls in a row.  With
    counts="self" and up to 32,768 ids it is one kernel whose blocks each count every id
    (N=1: every block's tokens begin ranks; R=2, N=3, H=20480: most blocks copy part of one
    token and own none), else the sort and the row copy as its programmatic dependent.
    H=264 takes 16-byte vectors, H=20480 rows of several slabs."""
    cfg = dict(cfg)
    cap_frac = cfg.pop("cap_frac", None)
    R, N, E, K, H = cfg["R"], cfg["N"], cfg["E"], cfg["K"], cfg["H"]
    inp = wl.make_ep(dict(cfg, routing="uniform", dtype="bf16"), seed=N + 7)
    inp.topk_idx[:, ::6, K - 1] = -1
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    if counts == "layout":
        B.check(plan.layout())
    cap = R * N * K if cap_frac is None else int(R * N * K * cap_frac)
    nb = R if rank_major else E
    dev = "cuda"
    want, st = (oracle.dispatch_ll_rank_major if rank_major else oracle.dispatch_ll)(
        wl.bf16_bits(inp.x), inp.topk_idx, E, recv_capacity=cap)
    n = min(want["num_recv"], cap)
    keys = ("dest_offsets", "dest_src_offsets") if rank_major else ("expert_offsets",
                                                                    "expert_src_offsets")
    for rep in range(3):
        boff = torch.full((nb + 1,), -3, dtype=torch.int32, device=dev)
        bsoff = torch.full((nb, R), -3, dtype=torch.int32, device=dev)
        src = torch.full((max(cap, 1),), -3, dtype=torch.int32, device=dev)
        slot = torch.full((R, N, K), -3, dtype=torch.int32, device=dev)
        rx = torch.zeros((max(cap, 1), H), dtype=torch.bfloat16, device=dev)
        plan.dev_err.zero_()
        ntpe = plan.num_tokens_per_expert if counts == "layout" else None
        B.check(B.mp_dispatch_ll(R, N, K, E, H, B.MP_BF16, rank_major, plan.x, None, plan.topk_idx,
                                 ntpe, cap, boff, bsoff, src, slot, rx, None, plan.dev_err))
        torch.cuda.synchronize()
        assert plan.device_error() == st, rep
        assert np.array_equal(boff.cpu().numpy(), want[keys[0]]), rep
        assert np.array_equal(bsoff.cpu().numpy(), want[keys[1]]), rep
        assert np.array_equal(slot.cpu().numpy(), want["slot_row"]), rep
        assert np.array_equal(src[:n].cpu().numpy(), want["recv_src_token"]), rep
        assert np.array_equal(wl.bf16_bits(rx[:n]), want["recv_x"]), rep
    assert (st == 0) == (cap_frac is None)


def test_low_latency_one_call_dispatch_replays_as_a_cuda_graph():
    """mp_dispatch_ll + mp_combine_ll captured once and replayed (the programmatic
    dependency between the sort and the row copy is captured with them)."""
    R, N, E, K, H = 4, 96, 32, 4, 136
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=33)
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    cap = R * N * K
    dev = "cuda"
    eoff = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    esoff = torch.zeros((E, R), dtype=torch.int32, device=dev)
    src = torch.zeros(cap, dtype=torch.int32, device=dev)
    slot = torch.zeros((R, N, K), dtype=torch.int32, device=dev)
    rx = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
    out = torch.zeros((R, N, H), dtype=torch.bfloat16, device=dev)

    def step():
        B.check(B.mp_dispatch_ll(R, N, K, E, H, B.MP_BF16, 0, plan.x, None, plan.topk_idx, None,
                                 cap, eoff, esoff, src, slot, rx, None, plan.dev_err))
        B.check(B.mp_combine_ll(R, N, K, H, rx, cap, slot, plan.topk_weights, out,
                                plan.dev_err))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    ll, st = oracle.dispatch_ll(wl.bf16_bits(inp.x), inp.topk_idx, E)
    comb, st2 = oracle.combine_ll(ll["recv_x"], ll["slot_row"], inp.topk_weights)
    assert st == st2 == 0
    n = ll["num_recv"]
    for _ in range(3):
        rx.zero_()
        out.zero_()
        slot.fill_(-3)
        graph.replay()
        torch.cuda.synchronize()
        assert plan.device_error() == 0
        assert np.array_equal(slot.cpu().numpy(), ll["slot_row"])
        assert np.array_equal(wl.bf16_bits(rx[:n]), ll["recv_x"])
        assert_bf16_close(wl.bf16_bits(out), comb, "combine_ll after replay")


@pytest.mark.parametrize("H", [384, 4096], ids=["vector_copy", "bulk_copy"])
def test_low_latency_one_call_dispatch_e4m3_with_scales(H):
    """e4m3 rows with their scales through mp_dispatch_ll; rows of 4 KB take the bulk
    copies of the one-kernel dispatch."""
    R, N, E, K = 4, 200, 32, 4
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="e4m3"), seed=32)
    plan = EPPlan(R, N, K, E, H, "e4m3")
    plan.load(inp)
    cap = R * N * K
    dev = "cuda"
    eoff = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    esoff = torch.zeros((E, R), dtype=torch.int32, device=dev)
    src = torch.zeros(cap, dtype=torch.int32, device=dev)
    slot = torch.zeros((R, N, K), dtype=torch.int32, device=dev)
    rx = torch.zeros((cap, H), dtype=torch.uint8, device=dev)
    rs = torch.zeros((cap, H // 128), dtype=torch.float32, device=dev)
    B.check(B.mp_dispatch_ll(R, N, K, E, H, B.MP_E4M3, 0, plan.x, plan.x_scales, plan.topk_idx,
                             None, cap, eoff, esoff, src, slot, rx, rs, plan.dev_err))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    payload = np.concatenate([wl.u8_bits(inp.x), inp.x_scales.numpy().view(np.uint8)], axis=-1)
    ll, st = oracle.dispatch_ll(payload, inp.topk_idx, E)
    assert st == 0
    n = ll["num_recv"]
    assert np.array_equal(slot.cpu().numpy(), ll["slot_row"])
    assert np.array_equal(src[:n].cpu().numpy(), ll["recv_src_token"])
    assert np.array_equal(rx[:n].cpu().numpy(), ll["recv_x"][:, :H])
    assert np.array_equal(rs[:n].cpu().numpy().view(np.uint8), ll["recv_x"][:, H:])


LL_QUANT = [dict(R=8, N=128, E=256, K=8, H=7168), dict(R=5, N=77, E=20, K=6, H=384),
            dict(R=3, N=300, E=9, K=9, H=256), dict(R=4, N=500, E=16, K=4, H=128, cap_frac=0.5),
            dict(R=2, N=50, E=64, K=32, H=128), dict(R=4, N=0, E=16, K=4, H=128)]


@pytest.mark.parametrize("cfg", LL_QUANT, ids=lambda c: "R%(R)d_N%(N)d_E%(E)d_K%(K)d_H%(H)d" % c
                         + ("_cap" if "cap_frac" in c else ""))
@pytest.mark.parametrize("rank_major", [0, 1], ids=["expert_major", "rank_major"])
@pytest.mark.parametrize("fmt", ["e4m3", "mxfp8", "mxfp4"])
@pytest.mark.parametrize("call", ["one_call", "rows"])
def test_low_latency_quantised_dispatch_matches_oracle(cfg, rank_major, fmt, call):
    """The low-latency dispatch with the quantisation in the row copy -- mp_dispatch_ll_quant
    (one kernel that counts, places and quantises up to 16,384 ids, else the sort and then
    the quantising copy as its programmatic dependent) or the LL offsets followed by
    mp_dispatch_ll_rows_quant -- against the oracle's composition: every token
    row quantised by the oracle (codes and scales), then the oracle's LL layout of those
    bytes; bit for bit, two calls in a row, with all-zero, tiny and wide-range blocks."""
    cfg = dict(cfg)
    cap_frac = cfg.pop("cap_frac", None)
    R, N, E, K, H = cfg["R"], cfg["N"], cfg["E"], cfg["K"], cfg["H"]
    f = QFMT[fmt]
    qcode = {"e4m3": B.MP_Q_E4M3, "mxfp8": B.MP_Q_MXFP8, "mxfp4": B.MP_Q_MXFP4}[fmt]
    inp = wl.make_ep(dict(cfg, routing="uniform", dtype="bf16"), seed=N + 11)
    if N > 0:
        inp.topk_idx[:, ::5, K - 1] = -1
        inp.x = _special_blocks(inp.x.reshape(R * N, H), f["block"]).reshape(R, N, H)
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    cap = R * N * K if cap_frac is None else int(R * N * K * cap_frac)
    q, sc, st = getattr(oracle, f["quant"])(wl.bf16_bits(inp.x))
    assert st == 0
    ncode = f["qcols"](H)
    nsb = (H // f["block"]) * sc.itemsize  # scale bytes per row
    payload = np.concatenate([q.reshape(R, N, ncode),
                              np.ascontiguousarray(sc).view(np.uint8).reshape(R, N, nsb)],
                             axis=-1)
    want, st = (oracle.dispatch_ll_rank_major if rank_major else oracle.dispatch_ll)(
        payload, inp.topk_idx, E, recv_capacity=cap)
    n = min(want["num_recv"], cap)
    keys = ("dest_offsets", "dest_src_offsets") if rank_major else ("expert_offsets",
                                                                    "expert_src_offsets")
    nb = R if rank_major else E
    dev = "cuda"
    for rep in range(2):
        boff = torch.full((nb + 1,), -3, dtype=torch.int32, device=dev)
        bsoff = torch.full((nb, R), -3, dtype=torch.int32, device=dev)
        src = torch.full((max(cap, 1),), -3, dtype=torch.int32, device=dev)
        slot = torch.full((R, N, K), -3, dtype=torch.int32, device=dev)
        rq = torch.zeros((max(cap, 1), ncode), dtype=torch.uint8, device=dev)
        rs = torch.zeros((max(cap, 1), H // f["block"]), dtype=f["sdt"], device=dev)
        plan.dev_err.zero_()
        if call == "one_call":
            B.check(B.mp_dispatch_ll_quant(R, N, K, E, H, qcode, rank_major, plan.x, plan.topk_idx,
                                           None, cap, boff, bsoff, src, slot, rq, rs,
                                           plan.dev_err))
        else:
            off = B.mp_dispatch_ll_offsets_rank_major if rank_major else B.mp_dispatch_ll_offsets
            B.check(off(R, N, K, E, plan.topk_idx, None, cap, boff, bsoff, src, slot,
                        plan.dev_err))
            B.check(B.mp_dispatch_ll_rows_quant(R, N, K, H, qcode, plan.x, slot, cap, rq, rs))
        torch.cuda.synchronize()
        assert plan.device_error() == st, rep
        assert np.array_equal(boff.cpu().numpy(), want[keys[0]]), rep
        assert np.array_equal(bsoff.cpu().numpy(), want[keys[1]]), rep
        assert np.array_equal(slot.cpu().numpy(), want["slot_row"]), rep
        assert np.array_equal(src[:n].cpu().numpy(), want["recv_src_token"]), rep
        assert np.array_equal(rq[:n].cpu().numpy(), want["recv_x"][:n, :ncode]), rep
        assert np.array_equal(rs[:n].contiguous().view(torch.uint8).cpu().numpy(),
                              want["recv_x"][:n, ncode:]), rep
    assert (st == 0) == (cap_frac is None)


def test_low_latency_offsets_flag_bad_ids_when_counting_themselves():
    R, N, E, K = 4, 50, 16, 3
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=64, routing="uniform", dtype="bf16"), seed=9)
    inp.topk_idx[1, 3, 0] = E + 5
    inp.topk_idx[2, 7, 2] = -4
    dev = "cuda"
    cap = R * N * K
    topk = torch.from_numpy(inp.topk_idx).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    eoff = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    esoff = torch.zeros((E, R), dtype=torch.int32, device=dev)
    src = torch.zeros(cap, dtype=torch.int32, device=dev)
    slot = torch.zeros((R, N, K), dtype=torch.int32, device=dev)
    B.check(B.mp_dispatch_ll_offsets(R, N, K, E, topk, None, cap, eoff, esoff, src, slot, err))
    torch.cuda.synchronize()
    assert int(err.item()) == B.MP_ERR_BAD_EXPERT
    ll, st = oracle.dispatch_ll(np.zeros((R, N, 16), np.uint8), inp.topk_idx, E)
    assert st == 0
    assert np.array_equal(slot.cpu().numpy(), ll["slot_row"])
    assert np.array_equal(eoff.cpu().numpy(), ll["expert_offsets"])


@pytest.mark.parametrize("cfg", [dict(R=4, N=50, E=16, K=3, H=64),      # one kernel
                                 dict(R=4, N=3000, E=16, K=3, H=64)],  # sort + row copy
                         ids=["fused", "sort_then_copy"])
def test_low_latency_one_call_dispatch_flags_bad_ids(cfg):
    """Ids outside [-1, E) through mp_dispatch_ll counting itself: MP_ERR_BAD_EXPERT, no row
    for them, every other entry placed as the oracle places it."""
    R, N, E, K, H = cfg["R"], cfg["N"], cfg["E"], cfg["K"], cfg["H"]
    inp = wl.make_ep(dict(cfg, routing="uniform", dtype="bf16"), seed=19)
    inp.topk_idx[1, 3, 0] = E + 5
    inp.topk_idx[2, 7, 2] = -4
    inp.topk_idx[0, 0, 1] = -1
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    cap = R * N * K
    dev = "cuda"
    eoff = torch.full((E + 1,), -3, dtype=torch.int32, device=dev)
    esoff = torch.full((E, R), -3, dtype=torch.int32, device=dev)
    src = torch.full((cap,), -3, dtype=torch.int32, device=dev)
    slot = torch.full((R, N, K), -3, dtype=torch.int32, device=dev)
    rx = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
    B.check(B.mp_dispatch_ll(R, N, K, E, H, B.MP_BF16, 0, plan.x, None, plan.topk_idx, None,
                             cap, eoff, esoff, src, slot, rx, None, plan.dev_err))
    torch.cuda.synchronize()
    assert plan.device_error() == B.MP_ERR_BAD_EXPERT
    ll, st = oracle.dispatch_ll(wl.bf16_bits(inp.x), inp.topk_idx, E)
    assert st == 0  # the oracle treats ids outside [0, E) as "no row" without a status
    n = ll["num_recv"]
    assert slot[1, 3, 0].item() == -1 and slot[2, 7, 2].item() == -1
    assert np.array_equal(slot.cpu().numpy(), ll["slot_row"])
    assert np.array_equal(eoff.cpu().numpy(), ll["expert_offsets"])
    assert np.array_equal(esoff.cpu().numpy(), ll["expert_src_offsets"])
    assert np.array_equal(src[:n].cpu().numpy(), ll["recv_src_token"])
    assert np.array_equal(wl.bf16_bits(rx[:n]), ll["recv_x"])


@pytest.mark.parametrize("wide", [False, True], ids=["16B", "32B"])
def test_allgatherv_multi_matches_per_tensor_oracle(wide):
    """Tensors whose bytes all split into 32-byte vectors take the wide path; a
    144-byte-row tensor with an odd row count forces 16-byte vectors."""
    R, sizes = 5, [7, 0, 130, 1, 33]
    S = sum(sizes)
    g = torch.Generator().manual_seed(5)
    data = torch.randint(0, 256, (S, 2048), generator=g, dtype=torch.uint8)      # e.g. packed fp4
    scales = torch.randint(0, 256, (S, 16 * 8), generator=g, dtype=torch.uint8)  # 128-byte rows
    hid = torch.randn((S, 72), generator=g).to(torch.bfloat16)                    # 144-byte rows
    ins = [data, scales] if wide else [data, scales, hid]
    outs = [torch.zeros((R,) + tuple(t.shape), dtype=t.dtype, device="cuda") for t in ins]
    row_bytes = [t[0].nbytes for t in ins]
    B.check(B.mp_allgatherv_multi(R, row_bytes, sizes, [t.cuda() for t in ins], outs))
    torch.cuda.synchronize()
    for t, o in zip(ins, outs):
        want, st = oracle.allgatherv(t.view(torch.uint8).numpy(), sizes, R)
        assert st == 0
        assert np.array_equal(o.cpu().view(torch.uint8).numpy(), want)


def _special_blocks(x: torch.Tensor, block: int) -> torch.Tensor:
    """Plant an all-zero, a tiny, a large and a wide-range scale block in a [S][H] tensor."""
    x = x.float()
    S, H = x.shape
    x[0, :block] = 0.0
    if S > 1:
        x[1, block:2 * block] = 2.0**-130
    x[S - 1, :] *= 300.0
    x[S // 2, :32] *= torch.exp2(torch.arange(32, dtype=torch.float32) - 16)
    return x.to(torch.bfloat16)


# Quantised formats: scale block, code bytes per row, scale dtype, the gather and
# dispatch entry points, and the oracle's quantiser (codes, scales, status).
QFMT = {
    "e4m3": dict(block=128, qcols=lambda H: H, sdt=torch.float32,
                 gather="mp_allgatherv_e4m3", disp="mp_dispatch_rows_e4m3", quant="quantize_e4m3"),
    "mxfp8": dict(block=32, qcols=lambda H: H, sdt=torch.uint8,
                  gather="mp_allgatherv_mxfp8", disp="mp_dispatch_rows_mxfp8",
                  quant="quantize_mxfp8"),
    "mxfp4": dict(block=32, qcols=lambda H: H // 2, sdt=torch.uint8,
                  gather="mp_allgatherv_mxfp4", disp="mp_dispatch_rows_mxfp4",
                  quant="quantize_mxfp4"),
}


def _oracle_quant(fmt: str, x: torch.Tensor):
    """Oracle codes and scales (scales as raw bytes) of bf16 rows."""
    q, sc, st = getattr(oracle, QFMT[fmt]["quant"])(wl.bf16_bits(x))
    assert st == 0
    return q, sc.view(np.uint8)


@pytest.mark.parametrize("fmt", sorted(QFMT))
@pytest.mark.parametrize("R,H,sizes", [(5, 256, [7, 0, 130, 1, 33]), (1, 128, [3]),
                                       (32, 128, [1] * 32), (3, 384, [0, 0, 0])],
                         ids=["R5_ragged", "R1", "R32", "empty"])
def test_allgatherv_quantised_equals_quantise_then_gather(fmt, R, H, sizes):
    f = QFMT[fmt]
    S = sum(sizes)
    x = wl.random_bf16((max(S, 1), H), seed=R * H)[:S]
    if S:
        x = _special_blocks(x, f["block"])
    out = torch.full((R, S, f["qcols"](H)), 0x5A, dtype=torch.uint8, device="cuda")
    osc = torch.zeros((R, S, H // f["block"]), dtype=f["sdt"], device="cuda")
    osc.view(torch.uint8).fill_(0x5A)
    B.check(getattr(B, f["gather"])(R, H, sizes, x.cuda(), out, osc))
    torch.cuda.synchronize()
    q, sc = _oracle_quant(fmt, x)
    want_q, st1 = oracle.allgatherv(q, sizes, R)
    want_s, st2 = oracle.allgatherv(sc, sizes, R)
    assert st1 == st2 == 0
    assert np.array_equal(out.cpu().numpy(), want_q)
    got_s = osc.cpu().view(torch.uint8).numpy()
    assert np.array_equal(got_s, want_s.reshape(got_s.shape))


def _offset_16(t: torch.Tensor) -> torch.Tensor:
    """A CUDA copy of t whose data starts 16 bytes past a 32-byte boundary."""
    buf = torch.zeros(t.numel() * t.element_size() + 48, dtype=torch.uint8, device="cuda")
    base = (-buf.data_ptr()) % 32 + 16
    out = buf[base:base + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
    out.copy_(t)
    assert out.data_ptr() % 32 == 16
    return out


@pytest.mark.parametrize("which", ["source", "output"])
@pytest.mark.parametrize("fmt", sorted(QFMT))
def test_quantising_copies_with_16_byte_aligned_buffers(fmt, which):
    """A source that is 16- but not 32-byte aligned takes the 8-channels-per-lane form;
    an FP8 output of that alignment the 16-channel one (32 channels per lane store 32
    code bytes at once)."""
    f = QFMT[fmt]
    R, N, E, K, H = 4, 300, 16, 4, 384
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=77)
    inp.x = _special_blocks(inp.x.reshape(R * N, H), f["block"]).reshape(R, N, H)
    plan = EPPlan(R, N, K, E, H)
    plan.load(inp)
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    xo = _offset_16(plan.x) if which == "source" else plan.x
    nsc = H // f["block"]
    rq = torch.zeros((plan.cap, f["qcols"](H)), dtype=torch.uint8, device="cuda")
    if which == "output":
        rq = _offset_16(rq)
    rs = torch.zeros((plan.cap, nsc), dtype=f["sdt"], device="cuda")
    B.check(getattr(B, f["disp"])(R, N, H, xo, plan.send_row, plan.cap, rq, rs))
    sizes = [5, 0, 17]
    S = sum(sizes)
    sh = plan.x.reshape(R * N, H)[:S]
    sh = _offset_16(sh) if which == "source" else sh.contiguous()
    gq = torch.zeros((3, S, f["qcols"](H)), dtype=torch.uint8, device="cuda")
    if which == "output":
        gq = _offset_16(gq)
    gs = torch.zeros((3, S, nsc), dtype=f["sdt"], device="cuda")
    B.check(getattr(B, f["gather"])(3, H, sizes, sh, gq, gs))
    torch.cuda.synchronize()
    q, sc = _oracle_quant(fmt, inp.x)
    payload = np.concatenate([q, sc], axis=-1)
    _, _, mask, _ = oracle.layout(inp.topk_idx, E)
    out, st2 = oracle.dispatch(payload, inp.topk_idx, inp.topk_weights, mask, E)
    assert st2 == 0
    n = out["num_recv"]
    qc = f["qcols"](H)
    assert np.array_equal(rq[:n].cpu().numpy(), out["recv_x"][:, :qc])
    assert np.array_equal(rs[:n].cpu().view(torch.uint8).numpy(), out["recv_x"][:, qc:])
    flat_q, flat_s = q.reshape(R * N, -1)[:S], sc.reshape(R * N, -1)[:S]
    for r in range(3):
        assert np.array_equal(gq[r].cpu().numpy(), flat_q)
        assert np.array_equal(gs[r].cpu().view(torch.uint8).numpy(), flat_s)


@pytest.mark.parametrize("fmt", sorted(QFMT))
def test_quantisers_on_random_bit_patterns(fmt):
    """67 M elements: random finite bf16 bit patterns, each scale block shifted by a random
    power of two so that scales span most of the fp32 range; every code and scale must
    equal the oracle's (R=1 gather = plain quantisation)."""
    f = QFMT[fmt]
    S, H = 16384, 4096
    rng = np.random.default_rng(61)
    bits = rng.integers(0, 1 << 16, (S, H), dtype=np.uint32).astype(np.uint16)
    bits &= np.uint16(0x807F) | np.uint16(0x3F80)      # exponent field below 0x7F8: finite
    shift = rng.integers(-110, 120, (S, H // f["block"]), dtype=np.int64).repeat(f["block"], 1)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float() * torch.exp2(
        torch.from_numpy(shift).float())
    x = torch.nan_to_num(x, posinf=3.0e38, neginf=-3.0e38).to(torch.bfloat16)
    out = torch.zeros((1, S, f["qcols"](H)), dtype=torch.uint8, device="cuda")
    osc = torch.zeros((1, S, H // f["block"]), dtype=f["sdt"], device="cuda")
    B.check(getattr(B, f["gather"])(1, H, [S], x.cuda(), out, osc))
    torch.cuda.synchronize()
    q, sc = _oracle_quant(fmt, x)
    assert np.array_equal(osc[0].cpu().view(torch.uint8).numpy(), sc)
    got = out[0].cpu().numpy()
    bad = np.argwhere(got != q)
    assert bad.size == 0, "first mismatches at %s" % bad[:5].tolist()


@pytest.mark.parametrize("fmt", sorted(QFMT))
def test_allgatherv_quantised_full_size(fmt):
    """The rsv shape (R=8, H=4096, sizes ~ U{0..16384}): every rank's copy equals the
    oracle's quantisation of the gathered rows."""
    f = QFMT[fmt]
    rsv = wl.CONFIGS["rsv"]
    R, H = rsv["R"], rsv["H"]
    sizes = np.random.default_rng(0).integers(0, rsv["max_rows"] + 1, size=R).tolist()
    S = sum(sizes)
    x = _special_blocks(wl.gathered_bf16(S, H, seed=3), f["block"])
    out = torch.zeros((R, S, f["qcols"](H)), dtype=torch.uint8, device="cuda")
    osc = torch.zeros((R, S, H // f["block"]), dtype=f["sdt"], device="cuda")
    B.check(getattr(B, f["gather"])(R, H, sizes, x.cuda(), out, osc))
    torch.cuda.synchronize()
    q, sc = _oracle_quant(fmt, x)
    q = torch.from_numpy(q).cuda()
    sc = torch.from_numpy(sc).cuda()
    osc = osc.view(torch.uint8)
    for r in range(R):
        assert torch.equal(out[r], q), "rank %d codes" % r
        assert torch.equal(osc[r], sc), "rank %d scales" % r


# ---------------------------------------------------------------------------
# full-size workloads (the benchmark's launch configuration)
# ---------------------------------------------------------------------------
def test_dsv3_full():
    inp = wl.make_ep("dsv3", seed=0)
    plan = run_gpu(inp)
    out = compare_ep(inp, plan)
    # order-sensitive combine at full size: random expert outputs
    y = wl.random_bf16_rows(out["num_recv"], inp.H, seed=5)
    B.check(plan.combine(y.cuda()))
    torch.cuda.synchronize()
    comb, st = oracle.combine(wl.bf16_bits(y), out["send_row"])
    assert st == 0 and plan.device_error() == 0
    assert_bf16_close(wl.bf16_bits(plan.out), comb, "dsv3 combine(y)")


def test_skew_full():
    inp = wl.make_ep("skew", seed=0)
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    rows = int(np.unpackbits(mask.view(np.uint8)).sum())
    y = wl.random_bf16_rows(rows, inp.H, seed=12)
    compare_ep(inp, run_gpu(inp, y=y.cuda()), y_bits=wl.bf16_bits(y),
               what="skew full combine(y)")


def test_fp8_full():
    inp = wl.make_ep("fp8", seed=0)
    _, _, mask, _ = oracle.layout(inp.topk_idx, inp.E)
    total = int(np.unpackbits(mask.view(np.uint8)).sum())
    y = wl.random_bf16_rows(total, inp.H, seed=99)
    plan = run_gpu(inp, y=y.cuda())
    compare_ep(inp, plan, y_bits=wl.bf16_bits(y), what="fp8 full combine(y)")


def test_rsv_full():
    """Reduce-scatterv of the full rsv workload against the oracle on every row, and the
    all-gatherv of its shards."""
    inp = wl.make_rsv("rsv", seed=0)
    R, H, sizes, S = inp.R, inp.H, inp.sizes.tolist(), inp.S
    plan = RSVPlan(R, H, sizes)
    plan.x.copy_(inp.x)
    plan.shards.copy_(inp.shards)
    B.check(plan.reducescatterv())
    B.check(plan.allgatherv())
    torch.cuda.synchronize()
    rs, st = oracle.reducescatterv(wl.bf16_bits(inp.x), sizes)
    assert st == 0
    assert_bf16_close(wl.bf16_bits(plan.rs_out), rs, "rsv full")
    ag, st = oracle.allgatherv(wl.bf16_bits(inp.shards), sizes, R)
    assert st == 0
    assert np.array_equal(wl.bf16_bits(plan.ag_out), ag)
