"""Buffer allocation and call sequencing around the C ABI (torch is used for
device memory and streams only; every computation is a library kernel).

``EPPlan`` owns the device buffers of one (R, N, K, E, H, dtype) problem and
runs mp_layout -> mp_dispatch -> mp_combine on them; ``RSVPlan`` does the same
for mp_reducescatterv / mp_allgatherv.
"""
from __future__ import annotations

import torch

from . import binding as B


def _i32(n, dev):
    return torch.zeros(n, dtype=torch.int32, device=dev)


class EPPlan:
    def __init__(self, R: int, N: int, K: int, E: int, H: int, dtype: str = "bf16",
                 recv_capacity: int | None = None, device="cuda"):
        if dtype not in ("bf16", "e4m3"):
            raise ValueError("dtype must be bf16 or e4m3")
        self.R, self.N, self.K, self.E, self.H, self.dtype = R, N, K, E, H, dtype
        self.device = torch.device(device)
        dev = self.device
        self.cap = R * N * min(R, K) if recv_capacity is None else int(recv_capacity)
        ws = B.mp_workspace_size(R, N, E)
        if ws == 0:
            raise ValueError("invalid problem shape R=%d N=%d E=%d" % (R, N, E))
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        self.dev_err = _i32(1, dev)
        # inputs
        self.topk_idx = torch.full((R, N, K), -1, dtype=torch.int32, device=dev)
        self.topk_weights = torch.zeros((R, N, K), dtype=torch.float32, device=dev)
        xdt = torch.bfloat16 if dtype == "bf16" else torch.float8_e4m3fn
        self.x = torch.zeros((R, N, H), dtype=xdt, device=dev)
        self.x_scales = (torch.zeros((R, N, H // B.SCALE_BLOCK), dtype=torch.float32, device=dev)
                         if dtype == "e4m3" else None)
        # layout outputs
        self.num_tokens_per_rank = _i32((R, R), dev)
        self.num_tokens_per_expert = _i32((R, E), dev)
        self.is_token_in_rank = torch.zeros((R, N), dtype=torch.int32, device=dev)
        # dispatch outputs
        c1 = max(self.cap, 1)
        self.recv_x = torch.zeros((c1, H), dtype=xdt, device=dev)
        self.recv_scales = (torch.zeros((c1, H // B.SCALE_BLOCK), dtype=torch.float32, device=dev)
                            if dtype == "e4m3" else None)
        self.recv_src_rank = _i32(c1, dev)
        self.recv_src_idx = _i32(c1, dev)
        self.recv_topk_idx = _i32((c1, K), dev)
        self.recv_topk_weights = torch.zeros((c1, K), dtype=torch.float32, device=dev)
        self.dest_offsets = _i32(R + 1, dev)
        self.rank_prefix = _i32((R, R), dev)
        self.num_recv_tokens_per_expert = _i32((R, E // R), dev)
        self.send_row = _i32((R, N, R), dev)
        # combine output
        self.out = torch.zeros((R, N, H), dtype=torch.bfloat16, device=dev)

    def load(self, inp, non_blocking: bool = False) -> None:
        """Copy a workloads.EPInputs (CPU tensors / arrays) into the device inputs."""
        self.topk_idx.copy_(torch.as_tensor(inp.topk_idx), non_blocking=non_blocking)
        self.topk_weights.copy_(torch.as_tensor(inp.topk_weights), non_blocking=non_blocking)
        self.x.copy_(inp.x, non_blocking=non_blocking)
        if self.x_scales is not None:
            self.x_scales.copy_(inp.x_scales, non_blocking=non_blocking)

    def layout(self, stream=None) -> int:
        return B.mp_layout(self.R, self.N, self.K, self.E, self.topk_idx,
                           self.num_tokens_per_rank, self.num_tokens_per_expert,
                           self.is_token_in_rank, self.dev_err, self.workspace, stream)

    def dispatch(self, stream=None) -> int:
        return B.mp_dispatch(
            self.R, self.N, self.K, self.E, self.H,
            B.MP_BF16 if self.dtype == "bf16" else B.MP_E4M3, self.x, self.x_scales,
            self.topk_idx, self.topk_weights, self.is_token_in_rank, self.num_tokens_per_rank,
            self.num_tokens_per_expert, self.cap, self.recv_x, self.recv_scales,
            self.recv_src_rank, self.recv_src_idx, self.recv_topk_idx, self.recv_topk_weights,
            self.dest_offsets, self.rank_prefix, self.num_recv_tokens_per_expert, self.send_row,
            self.dev_err, self.workspace, stream)

    def layout_and_offsets(self, stream=None) -> int:
        """mp_layout + mp_dispatch_offsets in one call (one cooperative launch when the
        problem fits one resident grid)."""
        return B.mp_layout_and_offsets(
            self.R, self.N, self.K, self.E, self.topk_idx, self.topk_weights, self.cap,
            self.num_tokens_per_rank, self.num_tokens_per_expert, self.is_token_in_rank,
            self.recv_src_rank, self.recv_src_idx, self.recv_topk_idx, self.recv_topk_weights,
            self.dest_offsets, self.rank_prefix, self.num_recv_tokens_per_expert, self.send_row,
            self.dev_err, self.workspace, stream)

    def layout_dispatch(self, stream=None) -> int:
        """The whole dispatch in one call (mp_layout_dispatch): layout, receive offsets
        and row copy, the copy launched as a programmatic dependent of the offsets."""
        return B.mp_layout_dispatch(
            self.R, self.N, self.K, self.E, self.H,
            B.MP_BF16 if self.dtype == "bf16" else B.MP_E4M3, self.x, self.x_scales,
            self.topk_idx, self.topk_weights, self.cap, self.num_tokens_per_rank,
            self.num_tokens_per_expert, self.is_token_in_rank, self.recv_x, self.recv_scales,
            self.recv_src_rank, self.recv_src_idx, self.recv_topk_idx, self.recv_topk_weights,
            self.dest_offsets, self.rank_prefix, self.num_recv_tokens_per_expert, self.send_row,
            self.dev_err, self.workspace, stream)

    def dispatch_offsets(self, stream=None) -> int:
        return B.mp_dispatch_offsets(
            self.R, self.N, self.K, self.E, self.topk_idx, self.topk_weights,
            self.is_token_in_rank, self.num_tokens_per_rank, self.num_tokens_per_expert,
            self.cap, self.recv_src_rank, self.recv_src_idx, self.recv_topk_idx,
            self.recv_topk_weights, self.dest_offsets, self.rank_prefix,
            self.num_recv_tokens_per_expert, self.send_row, self.dev_err, self.workspace, stream)

    def dispatch_rows(self, x: torch.Tensor | None = None, x_scales=None, recv_x=None,
                      recv_scales=None, stream=None) -> int:
        """Copy rows with the current send_row (default: this plan's own x / recv_x)."""
        x = self.x if x is None else x
        return B.mp_dispatch_rows(
            self.R, self.N, self.H, B.MP_BF16 if self.dtype == "bf16" else B.MP_E4M3, x,
            self.x_scales if x_scales is None else x_scales, self.send_row, self.cap,
            self.recv_x if recv_x is None else recv_x,
            self.recv_scales if recv_scales is None else recv_scales, stream)

    def combine(self, y: torch.Tensor | None = None, stream=None) -> int:
        """Combine y (default: recv_x, i.e. identity experts) back into self.out."""
        y = self.recv_x if y is None else y
        if y.dtype != torch.bfloat16 or y.dim() != 2 or y.shape[1] != self.H:
            raise ValueError("combine takes bf16 rows [rows][H] (an e4m3 plan needs its "
                             "expert outputs as y)")
        return B.mp_combine(self.R, self.N, self.H, y, y.shape[0], self.send_row, self.out,
                            self.dev_err, stream)

    def step(self, y: torch.Tensor | None = None, stream=None) -> None:
        """One pass of the hot path: layout -> dispatch -> combine as two calls (the whole
        dispatch in one call, then combine)."""
        B.check(self.layout_dispatch(stream), "mp_layout_dispatch")
        B.check(self.combine(y, stream), "mp_combine")

    def step_three_calls(self, y: torch.Tensor | None = None, stream=None) -> None:
        """The same pass as three calls: layout and receive offsets, row copy, combine."""
        B.check(self.layout_and_offsets(stream), "mp_layout_and_offsets")
        B.check(self.dispatch_rows(stream=stream), "mp_dispatch_rows")
        B.check(self.combine(y, stream), "mp_combine")

    def num_recv(self) -> int:
        return int(self.dest_offsets[self.R].item())

    def device_error(self) -> int:
        return int(self.dev_err.item())


class RSVPlan:
    def __init__(self, R: int, H: int, sizes, device="cuda"):
        self.R, self.H = R, H
        self.sizes = [int(s) for s in sizes]
        self.S = sum(self.sizes)
        dev = torch.device(device)
        self.x = torch.zeros((R, self.S, H), dtype=torch.bfloat16, device=dev)
        self.rs_out = torch.zeros((self.S, H), dtype=torch.bfloat16, device=dev)
        self.shards = torch.zeros((self.S, H), dtype=torch.bfloat16, device=dev)
        self.ag_out = torch.zeros((R, self.S, H), dtype=torch.bfloat16, device=dev)

    def reducescatterv(self, stream=None) -> int:
        return B.mp_reducescatterv(self.R, self.H, self.sizes, self.x, self.rs_out, stream)

    def allgatherv(self, stream=None) -> int:
        return B.mp_allgatherv(self.R, self.H * 2, self.sizes, self.shards, self.ag_out, stream)
