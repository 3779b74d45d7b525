"""CPU oracle for the MoE dispatch/combine path -- TEST INFRASTRUCTURE ONLY.

Thin numpy/ctypes wrapper around ``mp_oracle.c`` (plain single-threaded C,
built with ``-ffp-contract=off``).  Only the tests, the package smoke check
and the benchmark's CPU-baseline leg use this module; the library under
test never imports it and shares no code with it.

Every function follows the literal definition of its step; see the header
comment of ``mp_oracle.c`` for the passages cited and the readings taken
where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mp_oracle.c")
_LIB = os.path.join(_HERE, "libmp_oracle.so")

BAD_ARG = 1
CAPACITY = 4
BAD_EXPERT = 8


GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def compile_oracle(src: str, out: str) -> str:
    """Compile one copy of the oracle source with gcc (no GPU, no CUDA headers)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, src])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the default oracle library next to its source (if stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_oracle(_SRC, _LIB)
    return _LIB


class OracleLib:
    """One compiled copy of the oracle (the default build, or a test's own build)."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        L.oracle_layout.argtypes = [i32, i32, i32, i32, P, P, P, P]
        L.oracle_dispatch.argtypes = [i32, i32, i32, i32, i64, i32, P, P, P, P, P, i64,
                                      P, P, P, P, P, P, P, P, P, P]
        L.oracle_combine.argtypes = [i32, i32, i32, P, i64, P, P]
        L.oracle_reducescatterv.argtypes = [i32, i32, P, P, P]
        L.oracle_allgatherv.argtypes = [i32, i64, P, P, P]
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16_array.argtypes = [i64, P, P]
        L.oracle_f32_to_bf16_array.restype = None
        L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f32.restype = ctypes.c_float
        L.oracle_quantize_e4m3.argtypes = [i64, i32, P, P, P]
        L.oracle_quantize_e4m3.restype = ctypes.c_int
        L.oracle_recv_topk_global.argtypes = [i32, i32, i32, i32, P, P, P, P, ctypes.c_int32, P]
        L.oracle_recv_topk_global.restype = ctypes.c_int
        L.oracle_combine_weights.argtypes = [i32, i32, i32, P, i64, P, P]
        L.oracle_combine_weights.restype = ctypes.c_int
        L.oracle_quantize_mxfp8.argtypes = [i64, i32, P, P, P]
        L.oracle_quantize_mxfp8.restype = ctypes.c_int
        L.oracle_quantize_mxfp4.argtypes = [i64, i32, P, P, P]
        L.oracle_quantize_mxfp4.restype = ctypes.c_int
        L.oracle_f32_to_e2m1.argtypes = [ctypes.c_float]
        L.oracle_f32_to_e2m1.restype = ctypes.c_uint8
        L.oracle_e2m1_to_f32.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_to_f32.restype = ctypes.c_float
        L.oracle_dispatch_ll.argtypes = [i32, i32, i32, i32, i64, P, P, i64, P, P, P, P, P]
        L.oracle_dispatch_ll.restype = ctypes.c_int
        L.oracle_dispatch_ll_rank_major.argtypes = [i32, i32, i32, i32, i64, P, P, i64, P, P, P,
                                                    P, P]
        L.oracle_dispatch_ll_rank_major.restype = ctypes.c_int
        L.oracle_combine_ll.argtypes = [i32, i32, i32, i32, P, i64, P, P, P]
        L.oracle_combine_ll.restype = ctypes.c_int
        for f in ("oracle_layout", "oracle_dispatch", "oracle_combine",
                  "oracle_reducescatterv", "oracle_allgatherv"):
            getattr(L, f).restype = ctypes.c_int
        self.L = L
        self.path = path

    def layout(self, topk_idx: np.ndarray, E: int):
        """topk_idx int32 [R][N][K] -> (num_tokens_per_rank [R][R], num_tokens_per_expert
        [R][E], is_token_in_rank uint32 [R][N], status)."""
        topk_idx = _c(topk_idx, np.int32)
        R, N, K = topk_idx.shape
        ntpr = np.zeros((R, R), np.int32)
        ntpe = np.zeros((R, E), np.int32)
        mask = np.zeros((R, N), np.uint32)
        st = self.L.oracle_layout(R, N, K, E, _p(topk_idx), _p(ntpr), _p(ntpe), _p(mask))
        return ntpr, ntpe, mask, st

    def dispatch(self, x: np.ndarray, topk_idx: np.ndarray, topk_weights: np.ndarray,
                 is_token_in_rank: np.ndarray, E: int, x_scales: np.ndarray | None = None,
                 recv_capacity: int | None = None):
        """x [R][N][...] of any element type (rows copied as bytes).  Returns a dict of
        outputs (receive rows trimmed to the rows written) and the status."""
        x = np.ascontiguousarray(x)
        topk_idx = _c(topk_idx, np.int32)
        topk_weights = _c(topk_weights, np.float32)
        mask = _c(is_token_in_rank, np.uint32)
        R, N, K = topk_idx.shape
        row_shape = x.shape[2:]
        row_bytes = x.itemsize * int(np.prod(row_shape))
        if x_scales is not None:
            x_scales = _c(x_scales, np.float32)
            spr = x_scales.shape[-1]
        else:
            spr = 0
        total = int(np.unpackbits(mask.view(np.uint8)).sum()) if mask.size else 0
        cap = total if recv_capacity is None else int(recv_capacity)
        n1 = max(cap, 1)
        recv_x = np.zeros((n1,) + row_shape, x.dtype)
        recv_scales = np.zeros((n1, max(spr, 1)), np.float32)
        src_rank = np.full(n1, -7, np.int32)
        src_idx = np.full(n1, -7, np.int32)
        r_topk = np.full((n1, K), -7, np.int32)
        r_w = np.full((n1, K), -7.0, np.float32)
        dest_offsets = np.zeros(R + 1, np.int32)
        rank_prefix = np.zeros((R, R), np.int32)
        nrtpe = np.zeros((R, E // R), np.int32)
        send_row = np.zeros((R, N, R), np.int32)
        st = self.L.oracle_dispatch(
            R, N, K, E, row_bytes, spr, _p(x), _p(x_scales) if spr else None, _p(topk_idx),
            _p(topk_weights), _p(mask), cap, _p(recv_x), _p(recv_scales), _p(src_rank),
            _p(src_idx), _p(r_topk), _p(r_w), _p(dest_offsets), _p(rank_prefix), _p(nrtpe),
            _p(send_row))
        n = min(cap, total)
        out = dict(recv_x=recv_x[:n], recv_src_rank=src_rank[:n], recv_src_idx=src_idx[:n],
                   recv_topk_idx=r_topk[:n], recv_topk_weights=r_w[:n],
                   dest_offsets=dest_offsets, rank_prefix=rank_prefix,
                   num_recv_tokens_per_expert=nrtpe, send_row=send_row, num_recv=total)
        if spr:
            out["recv_scales"] = recv_scales[:n]
        return out, st

    def combine(self, y_bits: np.ndarray, send_row: np.ndarray):
        """y_bits uint16 (bf16 bit patterns) [rows][H]; send_row int32 [R][N][R].
        Returns (out uint16 [R][N][H], status)."""
        y_bits = _c(y_bits, np.uint16)
        send_row = _c(send_row, np.int32)
        R, N, _ = send_row.shape
        H = y_bits.shape[1]
        out = np.zeros((R, N, H), np.uint16)
        st = self.L.oracle_combine(R, N, H, _p(y_bits), y_bits.shape[0], _p(send_row), _p(out))
        return out, st

    def reducescatterv(self, in_bits: np.ndarray, sizes):
        """in_bits uint16 [R][S][H]; sizes length R.  Returns (out uint16 [S][H], status)."""
        in_bits = _c(in_bits, np.uint16)
        R, S, H = in_bits.shape
        sz = _c(np.asarray(sizes, np.int64), np.int64)
        assert sz.shape == (R,) and int(sz.sum()) == S
        out = np.zeros((S, H), np.uint16)
        st = self.L.oracle_reducescatterv(R, H, _p(sz), _p(in_bits), _p(out))
        return out, st

    def allgatherv(self, inp: np.ndarray, sizes, R: int):
        """inp [S][...] any dtype; sizes length R.  Returns (out [R][S][...], status)."""
        inp = np.ascontiguousarray(inp)
        S = inp.shape[0]
        sz = _c(np.asarray(sizes, np.int64), np.int64)
        assert sz.shape == (R,) and int(sz.sum()) == S
        row_bytes = inp.itemsize * int(np.prod(inp.shape[1:]))
        out = np.zeros((R,) + inp.shape, inp.dtype)
        st = self.L.oracle_allgatherv(R, row_bytes, _p(sz), _p(inp), _p(out))
        return out, st

    def bf16_to_f32(self, b: int) -> float:
        return self.L.oracle_bf16_to_f32(b)

    def f32_to_bf16(self, f: float) -> int:
        return self.L.oracle_f32_to_bf16(f)

    def f32_to_e4m3(self, f: float) -> int:
        return self.L.oracle_f32_to_e4m3(f)

    def e4m3_to_f32(self, b: int) -> float:
        return self.L.oracle_e4m3_to_f32(b)

    def quantize_e4m3(self, x_bits: np.ndarray):
        """x_bits uint16 (bf16 patterns) [..., H] -> (q uint8 [..., H], scales fp32
        [..., H/128], status)."""
        x_bits = _c(x_bits, np.uint16)
        H = x_bits.shape[-1]
        T = x_bits.size // H if H else 0
        q = np.zeros(x_bits.shape, np.uint8)
        sc = np.zeros(x_bits.shape[:-1] + (max(H // 128, 1),), np.float32)
        st = self.L.oracle_quantize_e4m3(T, H, _p(x_bits), _p(q), _p(sc))
        return q, sc, st

    def quantize_mxfp8(self, x_bits: np.ndarray):
        """x_bits uint16 (bf16 patterns) [..., H] -> (q uint8 [..., H], UE8M0 codes uint8
        [..., H/32], status)."""
        x_bits = _c(x_bits, np.uint16)
        H = x_bits.shape[-1]
        T = x_bits.size // H if H else 0
        q = np.zeros(x_bits.shape, np.uint8)
        codes = np.zeros(x_bits.shape[:-1] + (max(H // 32, 1),), np.uint8)
        st = self.L.oracle_quantize_mxfp8(T, H, _p(x_bits), _p(q), _p(codes))
        return q, codes, st

    def quantize_mxfp4(self, x_bits: np.ndarray):
        """x_bits uint16 (bf16 patterns) [..., H] -> (q uint8 [..., H/2] (two E2M1 codes
        per byte, even channel in the low nibble), UE8M0 codes uint8 [..., H/32], status)."""
        x_bits = _c(x_bits, np.uint16)
        H = x_bits.shape[-1]
        T = x_bits.size // H if H else 0
        q = np.zeros(x_bits.shape[:-1] + (max(H // 2, 1),), np.uint8)
        codes = np.zeros(x_bits.shape[:-1] + (max(H // 32, 1),), np.uint8)
        st = self.L.oracle_quantize_mxfp4(T, H, _p(x_bits), _p(q), _p(codes))
        return q, codes, st

    def f32_to_e2m1(self, f: float) -> int:
        return self.L.oracle_f32_to_e2m1(f)

    def e2m1_to_f32(self, c: int) -> float:
        return self.L.oracle_e2m1_to_f32(c)

    def recv_topk_global(self, topk_idx, E, disp: dict, sentinel: int):
        """Global expert ids of the receive rows of an oracle dispatch result."""
        topk_idx = _c(topk_idx, np.int32)
        R, N, K = topk_idx.shape
        T = int(disp["num_recv"])
        out = np.full((max(T, 1), K), -7, np.int32)
        src_rank = _c(disp["recv_src_rank"], np.int32)
        src_idx = _c(disp["recv_src_idx"], np.int32)
        offs = _c(disp["dest_offsets"], np.int32)
        st = self.L.oracle_recv_topk_global(R, N, K, E, _p(topk_idx), _p(src_rank), _p(src_idx),
                                            _p(offs), sentinel, _p(out))
        return out[:T], st

    def combine_weights(self, recv_topk_weights: np.ndarray, send_row: np.ndarray):
        """recv_topk_weights fp32 [rows][K], send_row [R][N][R] -> (fp32 [R][N][K], status)."""
        w = _c(recv_topk_weights, np.float32)
        send_row = _c(send_row, np.int32)
        R, N, _ = send_row.shape
        K = w.shape[1]
        out = np.zeros((R, N, K), np.float32)
        st = self.L.oracle_combine_weights(R, N, K, _p(w), w.shape[0], _p(send_row), _p(out))
        return out, st

    def dispatch_ll(self, x: np.ndarray, topk_idx: np.ndarray, E: int,
                    recv_capacity: int | None = None):
        """Expert-major low-latency dispatch of x [R][N][...] (bytes copied)."""
        x = np.ascontiguousarray(x)
        topk_idx = _c(topk_idx, np.int32)
        R, N, K = topk_idx.shape
        row_shape = x.shape[2:]
        row_bytes = x.itemsize * int(np.prod(row_shape))
        total = int(((topk_idx >= 0) & (topk_idx < E)).sum())
        cap = total if recv_capacity is None else int(recv_capacity)
        n1 = max(cap, 1)
        recv_x = np.zeros((n1,) + row_shape, x.dtype)
        src = np.full(n1, -7, np.int32)
        eoff = np.zeros(E + 1, np.int32)
        esoff = np.zeros((E, R), np.int32)
        slot = np.zeros((R, N, K), np.int32)
        st = self.L.oracle_dispatch_ll(R, N, K, E, row_bytes, _p(x), _p(topk_idx), cap,
                                       _p(recv_x), _p(src), _p(eoff), _p(esoff), _p(slot))
        n = min(cap, total)
        return dict(recv_x=recv_x[:n], recv_src_token=src[:n], expert_offsets=eoff,
                    expert_src_offsets=esoff, slot_row=slot, num_recv=total), st

    def dispatch_ll_rank_major(self, x: np.ndarray, topk_idx: np.ndarray, E: int,
                               recv_capacity: int | None = None):
        """Rank-major low-latency dispatch of x [R][N][...] (bytes copied)."""
        x = np.ascontiguousarray(x)
        topk_idx = _c(topk_idx, np.int32)
        R, N, K = topk_idx.shape
        row_shape = x.shape[2:]
        row_bytes = x.itemsize * int(np.prod(row_shape))
        total = int(((topk_idx >= 0) & (topk_idx < E)).sum())
        cap = total if recv_capacity is None else int(recv_capacity)
        n1 = max(cap, 1)
        recv_x = np.zeros((n1,) + row_shape, x.dtype)
        src = np.full(n1, -7, np.int32)
        doff = np.zeros(R + 1, np.int32)
        dsoff = np.zeros((R, R), np.int32)
        slot = np.zeros((R, N, K), np.int32)
        st = self.L.oracle_dispatch_ll_rank_major(R, N, K, E, row_bytes, _p(x), _p(topk_idx), cap,
                                                  _p(recv_x), _p(src), _p(doff), _p(dsoff),
                                                  _p(slot))
        n = min(cap, total)
        return dict(recv_x=recv_x[:n], recv_src_token=src[:n], dest_offsets=doff,
                    dest_src_offsets=dsoff, slot_row=slot, num_recv=total), st

    def combine_ll(self, y_bits: np.ndarray, slot_row: np.ndarray, topk_weights: np.ndarray):
        y_bits = _c(y_bits, np.uint16)
        slot_row = _c(slot_row, np.int32)
        w = _c(topk_weights, np.float32)
        R, N, K = slot_row.shape
        H = y_bits.shape[1]
        out = np.zeros((R, N, H), np.uint16)
        st = self.L.oracle_combine_ll(R, N, K, H, _p(y_bits), y_bits.shape[0], _p(slot_row),
                                      _p(w), _p(out))
        return out, st

    def f32_to_bf16_array(self, a: np.ndarray) -> np.ndarray:
        """Element-wise oracle narrowing of a binary32 array to bf16 bit patterns."""
        a = np.ascontiguousarray(a, np.float32)
        out = np.zeros(a.shape, np.uint16)
        self.L.oracle_f32_to_bf16_array(a.size, _p(a), _p(out))
        return out


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_default = None


def default() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def layout(*a, **k):
    return default().layout(*a, **k)


def dispatch(*a, **k):
    return default().dispatch(*a, **k)


def combine(*a, **k):
    return default().combine(*a, **k)


def reducescatterv(*a, **k):
    return default().reducescatterv(*a, **k)


def allgatherv(*a, **k):
    return default().allgatherv(*a, **k)


def f32_to_bf16_array(a):
    return default().f32_to_bf16_array(a)


def quantize_e4m3(x_bits):
    return default().quantize_e4m3(x_bits)


def recv_topk_global(topk_idx, E, disp, sentinel):
    return default().recv_topk_global(topk_idx, E, disp, sentinel)


def quantize_mxfp8(x_bits):
    return default().quantize_mxfp8(x_bits)


def quantize_mxfp4(x_bits):
    return default().quantize_mxfp4(x_bits)


def combine_weights(recv_topk_weights, send_row):
    return default().combine_weights(recv_topk_weights, send_row)


def dispatch_ll(x, topk_idx, E, recv_capacity=None):
    return default().dispatch_ll(x, topk_idx, E, recv_capacity)


def dispatch_ll_rank_major(x, topk_idx, E, recv_capacity=None):
    return default().dispatch_ll_rank_major(x, topk_idx, E, recv_capacity)


def combine_ll(y_bits, slot_row, topk_weights):
    return default().combine_ll(y_bits, slot_row, topk_weights)
