"""Thin ctypes binding of ``libmp_layout.so`` (the C ABI in include/mp_layout.h).

Argument marshalling only: every function takes torch CUDA tensors (device
memory), passes their device pointers and the current CUDA stream to the C
entry point of the same name and returns its status.  Every step of the path
runs in the library's CUDA kernels; there is no CPU fallback, and a missing
library or a CPU tensor raises at once.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

MP_OK = 0
MP_ERR_INVALID_ARG = 1
MP_ERR_CUDA = 2
MP_ERR_CAPACITY = 4
MP_ERR_BAD_EXPERT = 8
MP_ERR_TIMEOUT = 16
MP_BF16 = 0
MP_E4M3 = 1
SCALE_BLOCK = 128
# formats of the low-latency dispatch's in-kernel quantisation
MP_Q_E4M3 = 0
MP_Q_MXFP8 = 1
MP_Q_MXFP4 = 2

_lib = None


class MPError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: status %d (%s)" % (what or "mp_layout", status,
                                                 mp_status_string(status)))


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libmp_layout.so is not built (run __graft_entry__.build() or "
                               "python -m combine_mp_layout_gb300._build): the CUDA path is "
                               "required, there is no fallback")
        L = ctypes.CDLL(_build.LIB)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.mp_status_string.argtypes = [i32]
        L.mp_status_string.restype = ctypes.c_char_p
        L.mp_workspace_size.argtypes = [i32, i32, i32]
        L.mp_workspace_size.restype = ctypes.c_size_t
        L.mp_layout.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P]
        L.mp_dispatch.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i64,
                                  P, P, P, P, P, P, P, P, P, P, P, P, P]
        L.mp_dispatch_offsets.argtypes = [i32, i32, i32, i32, P, P, P, P, P, i64,
                                          P, P, P, P, P, P, P, P, P, P, P]
        L.mp_dispatch_rows.argtypes = [i32, i32, i32, i32, P, P, P, i64, P, P, P]
        L.mp_dispatch_rows_e4m3.argtypes = [i32, i32, i32, P, P, i64, P, P, P]
        L.mp_dispatch_rows_mxfp8.argtypes = [i32, i32, i32, P, P, i64, P, P, P]
        L.mp_dispatch_offsets_global.argtypes = [i32, i32, i32, i32, P, P, P, P, P, i64,
                                                 ctypes.c_int32, P, P, P, P, P, P, P, P, P, P, P]
        L.mp_combine_weights.argtypes = [i32, i32, i32, P, i64, P, P, P, P]
        L.mp_dispatch_ll_offsets.argtypes = [i32, i32, i32, i32, P, P, i64, P, P, P, P, P, P]
        L.mp_dispatch_ll_offsets_rank_major.argtypes = L.mp_dispatch_ll_offsets.argtypes
        L.mp_dispatch_ll_rows.argtypes = [i32, i32, i32, i32, i32, P, P, P, i64, P, P, P]
        L.mp_combine_ll.argtypes = [i32, i32, i32, i32, P, i64, P, P, P, P, P]
        L.mp_combine.argtypes = [i32, i32, i32, P, i64, P, P, P, P]
        L.mp_reducescatterv.argtypes = [i32, i32, P, P, P, P]
        L.mp_allgatherv.argtypes = [i32, i64, P, P, P, P]
        L.mp_allgatherv_e4m3.argtypes = [i32, i32, P, P, P, P, P]
        L.mp_allgatherv_mxfp8.argtypes = [i32, i32, P, P, P, P, P]
        L.mp_allgatherv_mxfp4.argtypes = [i32, i32, P, P, P, P, P]
        L.mp_dispatch_rows_mxfp4.argtypes = [i32, i32, i32, P, P, i64, P, P, P]
        L.mp_dispatch_rows_bulk.argtypes = [i32, i32, i32, i32, P, P, P, i64, P, P, P, P]
        L.mp_layout_and_offsets.argtypes = [i32, i32, i32, i32, P, P, i64] + [P] * 14
        L.mp_dispatch_noalloc.argtypes = [i32] * 6 + [P] * 7 + [i64] + [P] * 12
        L.mp_layout_dispatch.argtypes = [i32] * 6 + [P] * 4 + [i64] + [P] * 16
        L.mp_dispatch_ll_rows_quant.argtypes = [i32] * 5 + [P, P, i64, P, P, P]
        L.mp_dispatch_ll_quant.argtypes = [i32] * 7 + [P] * 3 + [i64] + [P] * 8
        L.mp_allgatherv_multi.argtypes = [i32, i32, P, P, P, P, P]
        L.mp_dispatch_ll.argtypes = [i32] * 7 + [P] * 4 + [i64] + [P] * 8
        for f in ("mp_layout", "mp_dispatch", "mp_dispatch_offsets", "mp_dispatch_rows",
                  "mp_dispatch_rows_e4m3", "mp_dispatch_rows_mxfp8", "mp_dispatch_offsets_global",
                  "mp_combine_weights",
                  "mp_dispatch_ll_offsets", "mp_dispatch_ll_offsets_rank_major",
                  "mp_dispatch_ll_rows", "mp_combine_ll",
                  "mp_combine", "mp_reducescatterv", "mp_allgatherv",
                  "mp_allgatherv_e4m3", "mp_allgatherv_mxfp8", "mp_allgatherv_mxfp4",
                  "mp_dispatch_rows_mxfp4", "mp_dispatch_rows_bulk",
                  "mp_layout_and_offsets", "mp_dispatch_noalloc", "mp_allgatherv_multi",
                  "mp_dispatch_ll", "mp_layout_dispatch", "mp_dispatch_ll_rows_quant",
                  "mp_dispatch_ll_quant"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _dev(t: torch.Tensor | None, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor (the library runs on the GPU only)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def check(status: int, what: str = "") -> int:
    if status != MP_OK:
        raise MPError(status, what)
    return status


def mp_status_string(status: int) -> str:
    return lib().mp_status_string(status).decode()


def mp_workspace_size(R: int, N: int, E: int) -> int:
    return int(lib().mp_workspace_size(R, N, E))


def mp_layout(R, N, K, E, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
              is_token_in_rank, dev_err, workspace, stream=None) -> int:
    return lib().mp_layout(R, N, K, E, _dev(topk_idx, "topk_idx"),
                           _dev(num_tokens_per_rank, "num_tokens_per_rank"),
                           _dev(num_tokens_per_expert, "num_tokens_per_expert"),
                           _dev(is_token_in_rank, "is_token_in_rank"),
                           _dev(dev_err, "dev_err"), _dev(workspace, "workspace"),
                           _stream(stream))


def mp_dispatch(R, N, K, E, H, dtype, x, x_scales, topk_idx, topk_weights, is_token_in_rank,
                num_tokens_per_rank, num_tokens_per_expert, recv_capacity, recv_x,
                recv_scales, recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, dev_err,
                workspace, stream=None) -> int:
    return lib().mp_dispatch(
        R, N, K, E, H, dtype, _dev(x, "x"), _dev(x_scales, "x_scales"),
        _dev(topk_idx, "topk_idx"), _dev(topk_weights, "topk_weights"),
        _dev(is_token_in_rank, "is_token_in_rank"),
        _dev(num_tokens_per_rank, "num_tokens_per_rank"),
        _dev(num_tokens_per_expert, "num_tokens_per_expert"), int(recv_capacity),
        _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"),
        _dev(recv_src_rank, "recv_src_rank"), _dev(recv_src_idx, "recv_src_idx"),
        _dev(recv_topk_idx, "recv_topk_idx"), _dev(recv_topk_weights, "recv_topk_weights"),
        _dev(dest_offsets, "dest_offsets"), _dev(rank_prefix, "rank_prefix"),
        _dev(num_recv_tokens_per_expert, "num_recv_tokens_per_expert"),
        _dev(send_row, "send_row"), _dev(dev_err, "dev_err"), _dev(workspace, "workspace"),
        _stream(stream))


def mp_dispatch_offsets(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                        num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                        recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                        dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, dev_err,
                        workspace, stream=None) -> int:
    return lib().mp_dispatch_offsets(
        R, N, K, E, _dev(topk_idx, "topk_idx"), _dev(topk_weights, "topk_weights"),
        _dev(is_token_in_rank, "is_token_in_rank"),
        _dev(num_tokens_per_rank, "num_tokens_per_rank"),
        _dev(num_tokens_per_expert, "num_tokens_per_expert"), int(recv_capacity),
        _dev(recv_src_rank, "recv_src_rank"), _dev(recv_src_idx, "recv_src_idx"),
        _dev(recv_topk_idx, "recv_topk_idx"), _dev(recv_topk_weights, "recv_topk_weights"),
        _dev(dest_offsets, "dest_offsets"), _dev(rank_prefix, "rank_prefix"),
        _dev(num_recv_tokens_per_expert, "num_recv_tokens_per_expert"),
        _dev(send_row, "send_row"), _dev(dev_err, "dev_err"), _dev(workspace, "workspace"),
        _stream(stream))


def mp_dispatch_rows(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x, recv_scales,
                     stream=None) -> int:
    return lib().mp_dispatch_rows(R, N, H, dtype, _dev(x, "x"), _dev(x_scales, "x_scales"),
                                  _dev(send_row, "send_row"), int(recv_capacity),
                                  _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"),
                                  _stream(stream))


def mp_layout_and_offsets(R, N, K, E, topk_idx, topk_weights, recv_capacity,
                          num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                          recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                          dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                          dev_err, workspace, stream=None) -> int:
    return lib().mp_layout_and_offsets(
        R, N, K, E, _dev(topk_idx, "topk_idx"), _dev(topk_weights, "topk_weights"),
        int(recv_capacity), _dev(num_tokens_per_rank, "num_tokens_per_rank"),
        _dev(num_tokens_per_expert, "num_tokens_per_expert"),
        _dev(is_token_in_rank, "is_token_in_rank"), _dev(recv_src_rank, "recv_src_rank"),
        _dev(recv_src_idx, "recv_src_idx"), _dev(recv_topk_idx, "recv_topk_idx"),
        _dev(recv_topk_weights, "recv_topk_weights"), _dev(dest_offsets, "dest_offsets"),
        _dev(rank_prefix, "rank_prefix"),
        _dev(num_recv_tokens_per_expert, "num_recv_tokens_per_expert"),
        _dev(send_row, "send_row"), _dev(dev_err, "dev_err"), _dev(workspace, "workspace"),
        _stream(stream))


def mp_layout_dispatch(R, N, K, E, H, dtype, x, x_scales, topk_idx, topk_weights, recv_capacity,
                       num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank, recv_x,
                       recv_scales, recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                       dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, dev_err,
                       workspace, stream=None) -> int:
    return lib().mp_layout_dispatch(
        R, N, K, E, H, dtype, _dev(x, "x"), _dev(x_scales, "x_scales"),
        _dev(topk_idx, "topk_idx"), _dev(topk_weights, "topk_weights"), int(recv_capacity),
        _dev(num_tokens_per_rank, "num_tokens_per_rank"),
        _dev(num_tokens_per_expert, "num_tokens_per_expert"),
        _dev(is_token_in_rank, "is_token_in_rank"), _dev(recv_x, "recv_x"),
        _dev(recv_scales, "recv_scales"), _dev(recv_src_rank, "recv_src_rank"),
        _dev(recv_src_idx, "recv_src_idx"), _dev(recv_topk_idx, "recv_topk_idx"),
        _dev(recv_topk_weights, "recv_topk_weights"), _dev(dest_offsets, "dest_offsets"),
        _dev(rank_prefix, "rank_prefix"),
        _dev(num_recv_tokens_per_expert, "num_recv_tokens_per_expert"),
        _dev(send_row, "send_row"), _dev(dev_err, "dev_err"), _dev(workspace, "workspace"),
        _stream(stream))


def mp_dispatch_offsets_global(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                               num_tokens_per_rank, num_tokens_per_expert, recv_capacity, sentinel,
                               recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                               dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                               dev_err, workspace, stream=None) -> int:
    return lib().mp_dispatch_offsets_global(
        R, N, K, E, _dev(topk_idx, "topk_idx"), _dev(topk_weights, "topk_weights"),
        _dev(is_token_in_rank, "is_token_in_rank"),
        _dev(num_tokens_per_rank, "num_tokens_per_rank"),
        _dev(num_tokens_per_expert, "num_tokens_per_expert"), int(recv_capacity), int(sentinel),
        _dev(recv_src_rank, "recv_src_rank"), _dev(recv_src_idx, "recv_src_idx"),
        _dev(recv_topk_idx, "recv_topk_idx"), _dev(recv_topk_weights, "recv_topk_weights"),
        _dev(dest_offsets, "dest_offsets"), _dev(rank_prefix, "rank_prefix"),
        _dev(num_recv_tokens_per_expert, "num_recv_tokens_per_expert"),
        _dev(send_row, "send_row"), _dev(dev_err, "dev_err"), _dev(workspace, "workspace"),
        _stream(stream))


def mp_combine_weights(R, N, K, recv_topk_weights, recv_rows, send_row, combined, dev_err,
                       stream=None) -> int:
    return lib().mp_combine_weights(R, N, K, _dev(recv_topk_weights, "recv_topk_weights"),
                                    int(recv_rows), _dev(send_row, "send_row"),
                                    _dev(combined, "combined_topk_weights"),
                                    _dev(dev_err, "dev_err"), _stream(stream))


def mp_dispatch_rows_bulk(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                          recv_scales, dev_err, stream=None) -> int:
    return lib().mp_dispatch_rows_bulk(R, N, H, dtype, _dev(x, "x"), _dev(x_scales, "x_scales"),
                                       _dev(send_row, "send_row"), int(recv_capacity),
                                       _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"),
                                       _dev(dev_err, "dev_err"), _stream(stream))


def mp_dispatch_rows_e4m3(R, N, H, x, send_row, recv_capacity, recv_x, recv_scales,
                          stream=None) -> int:
    return lib().mp_dispatch_rows_e4m3(R, N, H, _dev(x, "x"), _dev(send_row, "send_row"),
                                       int(recv_capacity), _dev(recv_x, "recv_x"),
                                       _dev(recv_scales, "recv_scales"), _stream(stream))


def mp_dispatch_rows_mxfp8(R, N, H, x, send_row, recv_capacity, recv_x, recv_scales,
                           stream=None) -> int:
    return lib().mp_dispatch_rows_mxfp8(R, N, H, _dev(x, "x"), _dev(send_row, "send_row"),
                                        int(recv_capacity), _dev(recv_x, "recv_x"),
                                        _dev(recv_scales, "recv_scales"), _stream(stream))


def mp_dispatch_rows_mxfp4(R, N, H, x, send_row, recv_capacity, recv_x, recv_scales,
                           stream=None) -> int:
    return lib().mp_dispatch_rows_mxfp4(R, N, H, _dev(x, "x"), _dev(send_row, "send_row"),
                                        int(recv_capacity), _dev(recv_x, "recv_x"),
                                        _dev(recv_scales, "recv_scales"), _stream(stream))


def mp_combine(R, N, H, y, y_rows, send_row, out, dev_err, stream=None) -> int:
    return lib().mp_combine(R, N, H, _dev(y, "y"), int(y_rows), _dev(send_row, "send_row"),
                            _dev(out, "out"), _dev(dev_err, "dev_err"), _stream(stream))


def _host_sizes(sizes):
    arr = (ctypes.c_int64 * len(sizes))(*[int(s) for s in sizes])
    return arr


def mp_reducescatterv(R, H, sizes, inp, out, stream=None) -> int:
    return lib().mp_reducescatterv(R, H, _host_sizes(sizes), _dev(inp, "in"), _dev(out, "out"),
                                   _stream(stream))


def mp_allgatherv(R, row_bytes, sizes, inp, out, stream=None) -> int:
    return lib().mp_allgatherv(R, int(row_bytes), _host_sizes(sizes), _dev(inp, "in"),
                               _dev(out, "out"), _stream(stream))


def mp_allgatherv_e4m3(R, H, sizes, inp, out, out_scales, stream=None) -> int:
    return lib().mp_allgatherv_e4m3(R, H, _host_sizes(sizes), _dev(inp, "in"), _dev(out, "out"),
                                    _dev(out_scales, "out_scales"), _stream(stream))


def mp_allgatherv_mxfp8(R, H, sizes, inp, out, out_scales, stream=None) -> int:
    return lib().mp_allgatherv_mxfp8(R, H, _host_sizes(sizes), _dev(inp, "in"), _dev(out, "out"),
                                     _dev(out_scales, "out_scales"), _stream(stream))


def mp_allgatherv_mxfp4(R, H, sizes, inp, out, out_scales, stream=None) -> int:
    return lib().mp_allgatherv_mxfp4(R, H, _host_sizes(sizes), _dev(inp, "in"), _dev(out, "out"),
                                     _dev(out_scales, "out_scales"), _stream(stream))


def mp_dispatch_noalloc(R, N, K, E, H, dtype, x, x_scales, topk_idx, topk_weights,
                        is_token_in_rank, num_tokens_per_rank, num_tokens_per_expert,
                        recv_capacity, recv_x, recv_scales, recv_src_rank, recv_src_idx,
                        recv_topk_idx, recv_topk_weights, dest_offsets, rank_prefix,
                        num_recv_tokens_per_expert, send_row, dev_err, stream=None) -> int:
    """mp_dispatch without a workspace, for callers that cannot allocate device memory
    (the scan's scratch is a fixed array inside the library; see the C header)."""
    f = lib().mp_dispatch_noalloc
    return f(R, N, K, E, H, dtype, _dev(x, "x"), _dev(x_scales, "x_scales"),
             _dev(topk_idx, "topk_idx"), _dev(topk_weights, "topk_weights"),
             _dev(is_token_in_rank, "is_token_in_rank"),
             _dev(num_tokens_per_rank, "num_tokens_per_rank"),
             _dev(num_tokens_per_expert, "num_tokens_per_expert"), int(recv_capacity),
             _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"),
             _dev(recv_src_rank, "recv_src_rank"), _dev(recv_src_idx, "recv_src_idx"),
             _dev(recv_topk_idx, "recv_topk_idx"), _dev(recv_topk_weights, "recv_topk_weights"),
             _dev(dest_offsets, "dest_offsets"), _dev(rank_prefix, "rank_prefix"),
             _dev(num_recv_tokens_per_expert, "num_recv_tokens_per_expert"),
             _dev(send_row, "send_row"), _dev(dev_err, "dev_err"), _stream(stream))


def mp_allgatherv_multi(R, row_bytes, sizes, inputs, outputs, stream=None) -> int:
    """All-gatherv of several tensors with the same per-rank row counts, one launch."""
    f = lib().mp_allgatherv_multi
    n = len(inputs)
    if len(outputs) != n or len(row_bytes) != n:
        raise ValueError("one row size and one output per input")
    rb = (ctypes.c_int64 * n)(*[int(b) for b in row_bytes])
    ins = (ctypes.c_void_p * n)(*[_dev(t, "in").value for t in inputs])
    outs = (ctypes.c_void_p * n)(*[_dev(t, "out").value for t in outputs])
    return f(R, n, rb, _host_sizes(sizes), ins, outs, _stream(stream))


def mp_dispatch_ll_offsets(R, N, K, E, topk_idx, num_tokens_per_expert, recv_capacity,
                           expert_offsets, expert_src_offsets, recv_src_token, slot_row, dev_err,
                           stream=None) -> int:
    return lib().mp_dispatch_ll_offsets(
        R, N, K, E, _dev(topk_idx, "topk_idx"), _dev(num_tokens_per_expert, "num_tokens_per_expert"),
        int(recv_capacity), _dev(expert_offsets, "expert_offsets"),
        _dev(expert_src_offsets, "expert_src_offsets"), _dev(recv_src_token, "recv_src_token"),
        _dev(slot_row, "slot_row"), _dev(dev_err, "dev_err"), _stream(stream))


def mp_dispatch_ll_offsets_rank_major(R, N, K, E, topk_idx, num_tokens_per_expert,
                                      recv_capacity, dest_offsets, dest_src_offsets,
                                      recv_src_token, slot_row, dev_err, stream=None) -> int:
    return lib().mp_dispatch_ll_offsets_rank_major(
        R, N, K, E, _dev(topk_idx, "topk_idx"), _dev(num_tokens_per_expert, "num_tokens_per_expert"),
        int(recv_capacity), _dev(dest_offsets, "dest_offsets"),
        _dev(dest_src_offsets, "dest_src_offsets"), _dev(recv_src_token, "recv_src_token"),
        _dev(slot_row, "slot_row"), _dev(dev_err, "dev_err"), _stream(stream))


def mp_dispatch_ll_rows(R, N, K, H, dtype, x, x_scales, slot_row, recv_capacity, recv_x,
                        recv_scales, stream=None) -> int:
    return lib().mp_dispatch_ll_rows(R, N, K, H, dtype, _dev(x, "x"), _dev(x_scales, "x_scales"),
                                     _dev(slot_row, "slot_row"), int(recv_capacity),
                                     _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"),
                                     _stream(stream))


def mp_dispatch_ll(R, N, K, E, H, dtype, rank_major, x, x_scales, topk_idx,
                   num_tokens_per_expert, recv_capacity, bin_offsets, bin_src_offsets,
                   recv_src_token, slot_row, recv_x, recv_scales, dev_err,
                   stream=None) -> int:
    return lib().mp_dispatch_ll(
        R, N, K, E, H, dtype, int(rank_major), _dev(x, "x"), _dev(x_scales, "x_scales"),
        _dev(topk_idx, "topk_idx"), _dev(num_tokens_per_expert, "num_tokens_per_expert"),
        int(recv_capacity), _dev(bin_offsets, "bin_offsets"),
        _dev(bin_src_offsets, "bin_src_offsets"), _dev(recv_src_token, "recv_src_token"),
        _dev(slot_row, "slot_row"), _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"),
        _dev(dev_err, "dev_err"), _stream(stream))


def mp_combine_ll(R, N, K, H, y, y_rows, slot_row, topk_weights, out, dev_err, stream=None) -> int:
    return lib().mp_combine_ll(R, N, K, H, _dev(y, "y"), int(y_rows), _dev(slot_row, "slot_row"),
                               _dev(topk_weights, "topk_weights"), _dev(out, "out"),
                               _dev(dev_err, "dev_err"), _stream(stream))


def mp_dispatch_ll_rows_quant(R, N, K, H, qformat, x, slot_row, recv_capacity, recv_x,
                              recv_scales, stream=None) -> int:
    """LL row copy with the quantisation in the kernel (qformat MP_Q_E4M3 / _MXFP8 /
    _MXFP4): bf16 token rows in, codes and scales at every slot row."""
    return lib().mp_dispatch_ll_rows_quant(R, N, K, H, int(qformat), _dev(x, "x"),
                                           _dev(slot_row, "slot_row"), int(recv_capacity),
                                           _dev(recv_x, "recv_x"),
                                           _dev(recv_scales, "recv_scales"), _stream(stream))


def mp_dispatch_ll_quant(R, N, K, E, H, qformat, rank_major, x, topk_idx, num_tokens_per_expert,
                         recv_capacity, bin_offsets, bin_src_offsets, recv_src_token, slot_row,
                         recv_x, recv_scales, dev_err, stream=None) -> int:
    """mp_dispatch_ll with the quantisation in the row copy."""
    return lib().mp_dispatch_ll_quant(
        R, N, K, E, H, int(qformat), int(rank_major), _dev(x, "x"), _dev(topk_idx, "topk_idx"),
        _dev(num_tokens_per_expert, "num_tokens_per_expert"), int(recv_capacity),
        _dev(bin_offsets, "bin_offsets"), _dev(bin_src_offsets, "bin_src_offsets"),
        _dev(recv_src_token, "recv_src_token"), _dev(slot_row, "slot_row"),
        _dev(recv_x, "recv_x"), _dev(recv_scales, "recv_scales"), _dev(dev_err, "dev_err"),
        _stream(stream))
