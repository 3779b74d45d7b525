"""Out-of-bounds writes, caught without a sanitizer: every buffer a call writes is
placed between guard regions filled with a known byte, the unused tail of each
receive buffer is pre-filled with it too, and after the calls every guard byte must
be unchanged.  Shapes are ragged (token counts off the tile size, rows of 144
bytes that take the 16-byte vector path) and include a too-small capacity, so the
kernels' clamps are exercised.  Values are checked elsewhere against the oracle;
here only where the kernels write."""
import math

import numpy as np
import pytest
import torch

from combine_mp_layout_gb300 import binding as B
from combine_mp_layout_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PAT = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` whose bytes sit between two guard regions; the
    tensor starts on a 256-byte boundary (the library's vector paths need 16 or 32)."""

    def __init__(self, shape, dtype, fill=None):
        self.n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * GUARD + self.n + 512,), PAT, dtype=torch.uint8, device="cuda")
        self.off = GUARD + (-(self.buf.data_ptr() + GUARD)) % 256
        self.t = self.buf[self.off:self.off + self.n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool((b[:self.off] == PAT).all() and (b[self.off + self.n:] == PAT).all())


def untouched_rows(t: torch.Tensor, first: int) -> bool:
    """Rows from `first` on still hold the guard byte (nothing was written there)."""
    rest = t[first:].contiguous().view(torch.uint8)
    return bool((rest == PAT).all().item())


def ep_buffers(R, N, K, E, H, cap, x_dtype=torch.bfloat16):
    g = {
        "ntpr": Guarded((R, R), torch.int32), "ntpe": Guarded((R, E), torch.int32),
        "mask": Guarded((R, N), torch.int32), "recv_x": Guarded((max(cap, 1), H), x_dtype),
        "rsr": Guarded((max(cap, 1),), torch.int32), "rsi": Guarded((max(cap, 1),), torch.int32),
        "rti": Guarded((max(cap, 1), K), torch.int32),
        "rtw": Guarded((max(cap, 1), K), torch.float32),
        "doff": Guarded((R + 1,), torch.int32), "rp": Guarded((R, R), torch.int32),
        "nrtpe": Guarded((R, E // R), torch.int32), "send": Guarded((R, N, R), torch.int32),
        "out": Guarded((R, N, H), torch.bfloat16), "err": Guarded((1,), torch.int32, 0),
    }
    ws = B.mp_workspace_size(R, N, E)
    g["ws"] = Guarded((ws,), torch.uint8, 0)
    return g


EP_SHAPES = [(3, 333, 12, 3, 72, None), (4, 300, 16, 4, 1024, None), (2, 129, 8, 2, 256, 0.5)]


@pytest.mark.parametrize("fused", ["fused", "two_calls", "one_call"])
@pytest.mark.parametrize("shape", EP_SHAPES, ids=lambda s: "R%d_N%d_E%d_K%d_H%d" % s[:5]
                         + ("_cap" if s[5] else ""))
def test_ep_path_writes_only_its_buffers(shape, fused):
    R, N, E, K, H, cap_frac = shape
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=R + N)
    topk = torch.from_numpy(inp.topk_idx).cuda()
    w = torch.from_numpy(inp.topk_weights).cuda()
    x = inp.x.cuda()
    T = int(np.count_nonzero(np.any((inp.topk_idx[..., None] // (E // R))
                                    == np.arange(R)[None, None, None, :], axis=2)))
    cap = R * N * min(R, K) if cap_frac is None else int(T * cap_frac)
    g = ep_buffers(R, N, K, E, H, cap)
    t = {k: v.t for k, v in g.items()}
    if fused == "one_call":
        B.check(B.mp_layout_dispatch(
            R, N, K, E, H, B.MP_BF16, x, None, topk, w, cap, t["ntpr"], t["ntpe"], t["mask"],
            t["recv_x"], None, t["rsr"], t["rsi"], t["rti"], t["rtw"], t["doff"], t["rp"],
            t["nrtpe"], t["send"], t["err"], t["ws"]))
    elif fused == "fused":
        B.check(B.mp_layout_and_offsets(
            R, N, K, E, topk, w, cap, t["ntpr"], t["ntpe"], t["mask"], t["rsr"], t["rsi"],
            t["rti"], t["rtw"], t["doff"], t["rp"], t["nrtpe"], t["send"], t["err"], t["ws"]))
        B.check(B.mp_dispatch_rows(R, N, H, B.MP_BF16, x, None, t["send"], cap, t["recv_x"],
                                   None))
    else:
        B.check(B.mp_layout(R, N, K, E, topk, t["ntpr"], t["ntpe"], t["mask"], t["err"], t["ws"]))
        B.check(B.mp_dispatch(R, N, K, E, H, B.MP_BF16, x, None, topk, w, t["mask"], t["ntpr"],
                              t["ntpe"], cap, t["recv_x"], None, t["rsr"], t["rsi"], t["rti"],
                              t["rtw"], t["doff"], t["rp"], t["nrtpe"], t["send"], t["err"],
                              t["ws"]))
    B.check(B.mp_combine(R, N, H, t["recv_x"], cap, t["send"], t["out"], t["err"]))
    torch.cuda.synchronize()
    assert int(t["err"].item()) == (0 if cap_frac is None else B.MP_ERR_CAPACITY)
    bad = [k for k, v in g.items() if not v.intact()]
    assert not bad, "guard bytes overwritten next to %s" % bad
    written = min(T, cap)
    for k in ("recv_x", "rsr", "rsi", "rti", "rtw"):
        assert untouched_rows(t[k], written), "%s written past its %d rows" % (k, written)


@pytest.mark.parametrize("fmt", ["e4m3", "mxfp8", "mxfp4"])
def test_quantising_copies_write_only_their_buffers(fmt):
    R, N, E, K, H = 3, 333, 12, 3, 384
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=5)
    topk = torch.from_numpy(inp.topk_idx).cuda()
    w = torch.from_numpy(inp.topk_weights).cuda()
    x = inp.x.cuda()
    cap = R * N * min(R, K)
    g = ep_buffers(R, N, K, E, H, cap)
    t = {k: v.t for k, v in g.items()}
    B.check(B.mp_layout_and_offsets(R, N, K, E, topk, w, cap, t["ntpr"], t["ntpe"], t["mask"],
                                    t["rsr"], t["rsi"], t["rti"], t["rtw"], t["doff"], t["rp"],
                                    t["nrtpe"], t["send"], t["err"], t["ws"]))
    torch.cuda.synchronize()
    T = int(t["doff"][R].item())
    qcols, blk = (H // 2, 32) if fmt == "mxfp4" else (H, 128 if fmt == "e4m3" else 32)
    sdt = torch.float32 if fmt == "e4m3" else torch.uint8
    rq = Guarded((cap, qcols), torch.uint8)
    rs = Guarded((cap, H // blk), sdt)
    B.check(getattr(B, "mp_dispatch_rows_" + fmt)(R, N, H, x, t["send"], cap, rq.t, rs.t))
    sizes = [7, 0, 130]
    S = sum(sizes)
    gq = Guarded((R, S, qcols), torch.uint8)
    gs = Guarded((R, S, H // blk), sdt)
    shards = x.reshape(R * N, H)[:S].contiguous()
    B.check(getattr(B, "mp_allgatherv_" + fmt)(R, H, sizes, shards, gq.t, gs.t))
    torch.cuda.synchronize()
    for name, gb in (("codes", rq), ("scales", rs), ("gathered codes", gq),
                     ("gathered scales", gs)):
        assert gb.intact(), "guard bytes overwritten next to the " + name
    assert untouched_rows(rq.t, T) and untouched_rows(rs.t, T)


def test_collectives_write_only_their_buffers():
    R, H, sizes = 5, 72, [7, 0, 130, 1, 33]
    S = sum(sizes)
    rin = wl.make_rsv(dict(R=R, H=H, sizes=sizes), seed=3)
    rs = Guarded((S, H), torch.bfloat16)
    ag = Guarded((R, S, H), torch.bfloat16)
    B.check(B.mp_reducescatterv(R, H, sizes, rin.x.cuda(), rs.t))
    B.check(B.mp_allgatherv(R, H * 2, sizes, rin.shards.cuda(), ag.t))
    data = torch.randint(0, 256, (S, 48), dtype=torch.uint8).cuda()
    scales = torch.randint(0, 256, (S, 32), dtype=torch.uint8).cuda()
    od = Guarded((R, S, 48), torch.uint8)
    osc = Guarded((R, S, 32), torch.uint8)
    B.check(B.mp_allgatherv_multi(R, [48, 32], sizes, [data, scales], [od.t, osc.t]))
    torch.cuda.synchronize()
    for name, gb in (("reducescatterv", rs), ("allgatherv", ag), ("multi data", od),
                     ("multi scales", osc)):
        assert gb.intact(), "guard bytes overwritten next to the " + name + " output"


@pytest.mark.parametrize("rank_major", [False, True], ids=["expert_major", "rank_major"])
def test_low_latency_path_writes_only_its_buffers(rank_major):
    R, N, E, K, H = 4, 77, 16, 3, 72
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=9)
    inp.topk_idx[:, ::5, 1] = -1
    topk = torch.from_numpy(inp.topk_idx).cuda()
    w = torch.from_numpy(inp.topk_weights).cuda()
    x = inp.x.cuda()
    total = int((inp.topk_idx >= 0).sum())
    cap = total - 10  # too small: the last rows are dropped, nothing past cap is written
    nb = R if rank_major else E
    off = Guarded((nb + 1,), torch.int32)
    soff = Guarded((nb, R), torch.int32)
    src = Guarded((cap,), torch.int32)
    slot = Guarded((R, N, K), torch.int32)
    rx = Guarded((cap, H), torch.bfloat16)
    y = wl.random_bf16((cap, H), seed=1).cuda()
    out = Guarded((R, N, H), torch.bfloat16)
    err = Guarded((1,), torch.int32, 0)
    f = B.mp_dispatch_ll_offsets_rank_major if rank_major else B.mp_dispatch_ll_offsets
    B.check(f(R, N, K, E, topk, None, cap, off.t, soff.t, src.t, slot.t, err.t))
    B.check(B.mp_dispatch_ll_rows(R, N, K, H, B.MP_BF16, x, None, slot.t, cap, rx.t, None))
    B.check(B.mp_combine_ll(R, N, K, H, y, cap, slot.t, w, out.t, err.t))
    torch.cuda.synchronize()
    assert int(err.t.item()) == B.MP_ERR_CAPACITY
    for name, gb in (("offsets", off), ("source offsets", soff), ("source tokens", src),
                     ("slots", slot), ("rows", rx), ("combine", out), ("error word", err)):
        assert gb.intact(), "guard bytes overwritten next to the " + name


@pytest.mark.parametrize("rank_major", [0, 1], ids=["expert_major", "rank_major"])
def test_one_call_low_latency_dispatch_writes_only_its_buffers(rank_major):
    """mp_dispatch_ll (the sort, then the row copy as its programmatic dependent) with a
    too-small capacity."""
    R, N, E, K, H = 4, 77, 16, 3, 72
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=10)
    inp.topk_idx[:, ::5, 1] = -1
    topk = torch.from_numpy(inp.topk_idx).cuda()
    x = inp.x.cuda()
    total = int((inp.topk_idx >= 0).sum())
    cap = total - 10
    nb = R if rank_major else E
    off = Guarded((nb + 1,), torch.int32)
    soff = Guarded((nb, R), torch.int32)
    src = Guarded((cap,), torch.int32)
    slot = Guarded((R, N, K), torch.int32)
    rx = Guarded((cap, H), torch.bfloat16)
    err = Guarded((1,), torch.int32, 0)
    for _ in range(2):
        B.check(B.mp_dispatch_ll(R, N, K, E, H, B.MP_BF16, rank_major, x, None, topk, None, cap,
                                 off.t, soff.t, src.t, slot.t, rx.t, None, err.t))
    torch.cuda.synchronize()
    assert int(err.t.item()) == B.MP_ERR_CAPACITY
    for name, gb in (("offsets", off), ("source offsets", soff), ("source tokens", src),
                     ("slots", slot), ("rows", rx), ("error word", err)):
        assert gb.intact(), "guard bytes overwritten next to the " + name


@pytest.mark.parametrize("fmt", ["e4m3", "mxfp8", "mxfp4"])
@pytest.mark.parametrize("rank_major", [0, 1], ids=["expert_major", "rank_major"])
def test_quantised_low_latency_dispatch_writes_only_its_buffers(fmt, rank_major):
    """mp_dispatch_ll_quant and mp_dispatch_ll_rows_quant with a too-small capacity."""
    R, N, E, K, H = 4, 77, 16, 3, 256
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=12)
    inp.topk_idx[:, ::5, 1] = -1
    topk = torch.from_numpy(inp.topk_idx).cuda()
    x = inp.x.cuda()
    total = int((inp.topk_idx >= 0).sum())
    cap = total - 10
    nb = R if rank_major else E
    qcode = {"e4m3": B.MP_Q_E4M3, "mxfp8": B.MP_Q_MXFP8, "mxfp4": B.MP_Q_MXFP4}[fmt]
    qcols, blk = (H // 2, 32) if fmt == "mxfp4" else (H, 128 if fmt == "e4m3" else 32)
    sdt = torch.float32 if fmt == "e4m3" else torch.uint8
    off = Guarded((nb + 1,), torch.int32)
    soff = Guarded((nb, R), torch.int32)
    src = Guarded((cap,), torch.int32)
    slot = Guarded((R, N, K), torch.int32)
    rq = Guarded((cap, qcols), torch.uint8)
    rs = Guarded((cap, H // blk), sdt)
    rq2 = Guarded((cap, qcols), torch.uint8)
    rs2 = Guarded((cap, H // blk), sdt)
    err = Guarded((1,), torch.int32, 0)
    B.check(B.mp_dispatch_ll_quant(R, N, K, E, H, qcode, rank_major, x, topk, None, cap, off.t,
                                   soff.t, src.t, slot.t, rq.t, rs.t, err.t))
    B.check(B.mp_dispatch_ll_rows_quant(R, N, K, H, qcode, x, slot.t, cap, rq2.t, rs2.t))
    torch.cuda.synchronize()
    assert int(err.t.item()) == B.MP_ERR_CAPACITY
    for name, gb in (("offsets", off), ("source offsets", soff), ("source tokens", src),
                     ("slots", slot), ("codes", rq), ("scales", rs), ("codes (rows call)", rq2),
                     ("scales (rows call)", rs2), ("error word", err)):
        assert gb.intact(), "guard bytes overwritten next to the " + name


def test_bulk_copy_dispatch_writes_only_its_buffers():
    R, N, E, K, H = 3, 333, 12, 3, 72
    inp = wl.make_ep(dict(R=R, N=N, E=E, K=K, H=H, routing="uniform", dtype="bf16"), seed=11)
    topk = torch.from_numpy(inp.topk_idx).cuda()
    w = torch.from_numpy(inp.topk_weights).cuda()
    cap = R * N * min(R, K)
    g = ep_buffers(R, N, K, E, H, cap)
    t = {k: v.t for k, v in g.items()}
    B.check(B.mp_layout_and_offsets(R, N, K, E, topk, w, cap, t["ntpr"], t["ntpe"], t["mask"],
                                    t["rsr"], t["rsi"], t["rti"], t["rtw"], t["doff"], t["rp"],
                                    t["nrtpe"], t["send"], t["err"], t["ws"]))
    torch.cuda.synchronize()
    T = int(t["doff"][R].item())
    small = T // 2  # the bulk copy must also stop at the capacity
    rx = Guarded((small, H), torch.bfloat16)
    B.check(B.mp_dispatch_rows_bulk(R, N, H, B.MP_BF16, inp.x.cuda(), None, t["send"], small,
                                    rx.t, None, t["err"]))
    torch.cuda.synchronize()
    assert rx.intact()
