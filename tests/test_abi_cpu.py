"""The C ABI without a GPU: the library builds, loads and exports every symbol
the header declares; the host-side argument checks and the workspace sizing
behave as documented.  No call here reaches a CUDA launch (every argument
set below fails a host check first, or the call is host-only)."""
import ctypes
import os
import re

import pytest

from combine_mp_layout_gb300 import _build, binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mp_layout.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return B.lib()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for f in ("mp_layout", "mp_dispatch", "mp_combine", "mp_reducescatterv", "mp_allgatherv",
              "mp_workspace_size", "mp_status_string"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    assert B.mp_status_string(0) == "ok"
    assert "capacity" in B.mp_status_string(B.MP_ERR_CAPACITY)
    assert "expert" in B.mp_status_string(B.MP_ERR_BAD_EXPERT)
    assert "timed out" in B.mp_status_string(B.MP_ERR_TIMEOUT)
    assert "invalid" in B.mp_status_string(B.MP_ERR_INVALID_ARG | B.MP_ERR_CAPACITY)


def test_workspace_size(L):
    # control block + per-rank count accumulators + tile records (flag + 2R counts)
    # for tiles of 128 tokens that never straddle two source ranks + the fused
    # kernel's two rank-totals buffers of 32 x 32 int32
    s = B.mp_workspace_size(8, 4096, 256)
    tiles = 8 * ((4096 + 127) // 128)
    base = 512 + 8 * (256 + 8) * 4 + tiles * (4 + 2 * 8 * 4) + 2 * 32 * 32 * 4
    assert base <= s < base + 4 * 256
    assert s % 256 == 0
    assert B.mp_workspace_size(2, 0, 8) > 0
    assert B.mp_workspace_size(0, 10, 8) == 0      # R < 1
    assert B.mp_workspace_size(33, 10, 66) == 0    # R > 32
    assert B.mp_workspace_size(4, 10, 6) == 0      # E % R != 0
    assert B.mp_workspace_size(4, -1, 8) == 0


FAKE = 0x10000  # never dereferenced: every call below fails its host checks first

# The argument-check tests pass fake device addresses.  Every set is invalid, so
# nothing launches; they still run only where no GPU is visible, so that a
# mistake in a test can never send a kernel to a fake address.
no_gpu = pytest.mark.skipif(
    __import__("torch").cuda.is_available(),
    reason="fake-pointer argument checks run only on a host without a visible GPU")


def _p(v=FAKE):
    return ctypes.c_void_p(v)


def layout_args(**kw):
    a = dict(R=2, N=8, K=2, E=8, topk=_p(), ntpr=_p(), ntpe=_p(), mask=_p(), err=_p(), ws=_p(),
             stream=_p(0))
    a.update(kw)
    return [a["R"], a["N"], a["K"], a["E"], a["topk"], a["ntpr"], a["ntpe"], a["mask"],
            a["err"], a["ws"], a["stream"]]


@no_gpu
@pytest.mark.parametrize("bad", [
    dict(R=0), dict(R=33, E=66), dict(N=-1), dict(K=0), dict(K=33), dict(E=7),
    dict(E=1), dict(E=9000), dict(ntpr=_p(0)), dict(err=_p(0)), dict(ws=_p(0)),
    dict(topk=_p(FAKE + 2)), dict(ws=_p(FAKE + 8)), dict(R=32, N=2**21, K=32, E=64),
])
def test_layout_rejects(L, bad):
    assert L.mp_layout(*layout_args(**bad)) == B.MP_ERR_INVALID_ARG


def dispatch_args(**kw):
    a = dict(R=2, N=8, K=2, E=8, H=64, dtype=B.MP_BF16, x=_p(), xs=_p(0), cap=32, rx=_p(),
             rs=_p(0), ws=_p(), err=_p())
    a.update(kw)
    P = _p()
    return [a["R"], a["N"], a["K"], a["E"], a["H"], a["dtype"], a["x"], a["xs"], P, P, P, P, P,
            a["cap"], a["rx"], a["rs"], P, P, P, P, P, P, P, P, a["err"], a["ws"], _p(0)]


@no_gpu
@pytest.mark.parametrize("bad", [
    dict(H=0), dict(H=60), dict(dtype=7), dict(dtype=B.MP_E4M3, xs=_p(), rs=_p(), H=64 + 8),
    dict(dtype=B.MP_E4M3), dict(xs=_p()), dict(cap=-1), dict(x=_p(FAKE + 4)),
    dict(rx=_p(FAKE + 8)), dict(err=_p(0)), dict(E=9), dict(x=_p(0)),
])
def test_dispatch_rejects(L, bad):
    assert L.mp_dispatch(*dispatch_args(**bad)) == B.MP_ERR_INVALID_ARG


@no_gpu
@pytest.mark.parametrize("args", [
    (0, 4, 64, _p(), 10, _p(), _p(), _p(), _p(0)),      # R < 1
    (2, 4, 60, _p(), 10, _p(), _p(), _p(), _p(0)),      # H % 8
    (2, 4, 64, _p(), -1, _p(), _p(), _p(), _p(0)),      # y_rows < 0
    (2, 4, 64, _p(FAKE + 4), 10, _p(), _p(), _p(), _p(0)),  # y misaligned
    (2, 4, 64, _p(), 10, _p(), _p(), _p(0), _p(0)),     # dev_err NULL
])
def test_combine_rejects(L, args):
    assert L.mp_combine(*args) == B.MP_ERR_INVALID_ARG


@no_gpu
def test_collectives_reject(L):
    sizes = (ctypes.c_int64 * 3)(1, -2, 3)
    assert L.mp_reducescatterv(3, 64, sizes, _p(), _p(), _p(0)) == B.MP_ERR_INVALID_ARG
    assert L.mp_allgatherv(3, 128, sizes, _p(), _p(), _p(0)) == B.MP_ERR_INVALID_ARG
    ok = (ctypes.c_int64 * 3)(1, 2, 3)
    assert L.mp_reducescatterv(3, 60, ok, _p(), _p(), _p(0)) == B.MP_ERR_INVALID_ARG
    assert L.mp_allgatherv(3, 100, ok, _p(), _p(), _p(0)) == B.MP_ERR_INVALID_ARG
    assert L.mp_reducescatterv(3, 64, None, _p(), _p(), _p(0)) == B.MP_ERR_INVALID_ARG
    assert L.mp_allgatherv(3, 128, ok, _p(FAKE + 8), _p(), _p(0)) == B.MP_ERR_INVALID_ARG
    assert L.mp_reducescatterv(0, 64, ok, _p(), _p(), _p(0)) == B.MP_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(L):
    import torch
    t = torch.zeros(16, dtype=torch.int32)
    with pytest.raises(TypeError):
        B.mp_combine(2, 4, 64, t, 1, t, t, t)


@no_gpu
def test_newer_entry_points_reject(L):
    """Host checks of the NEXT-row entry points (every argument set below is invalid)."""
    P, N0 = _p(), _p(0)
    L.mp_dispatch_rows_e4m3.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int64] + [ctypes.c_void_p] * 3
    assert L.mp_dispatch_rows_e4m3(2, 8, 100, P, P, 16, P, P, N0) == B.MP_ERR_INVALID_ARG  # H % 128
    assert L.mp_dispatch_rows_e4m3(2, 8, 128, _p(FAKE + 8), P, 16, P, P, N0) == B.MP_ERR_INVALID_ARG
    L.mp_dispatch_rows_mxfp8.argtypes = L.mp_dispatch_rows_e4m3.argtypes
    assert L.mp_dispatch_rows_mxfp8(2, 8, 48, P, P, 16, P, P, N0) == B.MP_ERR_INVALID_ARG  # H % 32
    assert L.mp_dispatch_rows_mxfp8(2, 8, 64, P, P, 16, P, N0, N0) == B.MP_ERR_INVALID_ARG  # scales
    L.mp_combine_weights.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_int64] + \
        [ctypes.c_void_p] * 4
    assert L.mp_combine_weights(2, 8, 0, P, 4, P, P, P, N0) == B.MP_ERR_INVALID_ARG      # K < 1
    assert L.mp_combine_weights(2, 8, 2, P, 4, P, P, N0, N0) == B.MP_ERR_INVALID_ARG     # dev_err
    L.mp_dispatch_ll_offsets.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int64] + [ctypes.c_void_p] * 6
    assert L.mp_dispatch_ll_offsets(2, 8, 2, 7, P, P, 16, P, P, P, P, P, N0) == B.MP_ERR_INVALID_ARG
    assert L.mp_dispatch_ll_offsets(2, 8, 33, 8, P, P, 16, P, P, P, P, P, N0) == \
        B.MP_ERR_INVALID_ARG  # K > MP_MAX_TOPK
    L.mp_dispatch_ll_offsets_rank_major.argtypes = L.mp_dispatch_ll_offsets.argtypes
    assert L.mp_dispatch_ll_offsets_rank_major(2, 8, 2, 7, P, P, 16, P, P, P, P, P, N0) == \
        B.MP_ERR_INVALID_ARG  # E % R
    assert L.mp_dispatch_ll_offsets_rank_major(2, 8, 2, 8, P, P, 16, P, P, P, P, N0, N0) == \
        B.MP_ERR_INVALID_ARG  # dev_err
    L.mp_combine_ll.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_int64] + \
        [ctypes.c_void_p] * 5
    assert L.mp_combine_ll(2, 8, 2, 60, P, 4, P, P, P, P, N0) == B.MP_ERR_INVALID_ARG   # H % 8
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    sizes = (ctypes.c_int64 * 2)(3, 4)
    rb = (ctypes.c_int64 * 2)(64, 40)
    L.mp_allgatherv_multi.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    assert L.mp_allgatherv_multi(2, 2, rb, sizes, arr, arr, N0) == B.MP_ERR_INVALID_ARG   # 40 % 16
    assert L.mp_allgatherv_multi(2, 9, rb, sizes, arr, arr, N0) == B.MP_ERR_INVALID_ARG   # > 8 tensors
    L.mp_allgatherv_e4m3.argtypes = [ctypes.c_int] * 2 + [ctypes.c_void_p] * 5
    L.mp_allgatherv_mxfp8.argtypes = L.mp_allgatherv_e4m3.argtypes
    assert L.mp_allgatherv_e4m3(2, 96, sizes, P, P, P, N0) == B.MP_ERR_INVALID_ARG     # H % 128
    assert L.mp_allgatherv_e4m3(33, 128, sizes, P, P, P, N0) == B.MP_ERR_INVALID_ARG   # R > 32
    assert L.mp_allgatherv_e4m3(2, 128, sizes, P, P, _p(FAKE + 2), N0) == B.MP_ERR_INVALID_ARG
    assert L.mp_allgatherv_mxfp8(2, 48, sizes, P, P, P, N0) == B.MP_ERR_INVALID_ARG    # H % 32
    assert L.mp_allgatherv_mxfp8(2, 64, sizes, P, N0, P, N0) == B.MP_ERR_INVALID_ARG   # out NULL
    L.mp_allgatherv_mxfp4.argtypes = L.mp_allgatherv_e4m3.argtypes
    assert L.mp_allgatherv_mxfp4(2, 80, sizes, P, P, P, N0) == B.MP_ERR_INVALID_ARG    # H % 32
    assert L.mp_allgatherv_mxfp4(2, 64, sizes, _p(FAKE + 8), P, P, N0) == B.MP_ERR_INVALID_ARG
    L.mp_dispatch_rows_mxfp4.argtypes = L.mp_dispatch_rows_e4m3.argtypes
    assert L.mp_dispatch_rows_mxfp4(2, 8, 48, P, P, 16, P, P, N0) == B.MP_ERR_INVALID_ARG  # H % 32
    assert L.mp_dispatch_rows_mxfp4(2, 8, 64, P, N0, 16, P, P, N0) == B.MP_ERR_INVALID_ARG  # send_row
    L.mp_dispatch_rows_bulk.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 3 + \
        [ctypes.c_int64] + [ctypes.c_void_p] * 4
    assert L.mp_dispatch_rows_bulk(2, 8, 64, B.MP_BF16, P, N0, P, 16, P, N0, N0, N0) == \
        B.MP_ERR_INVALID_ARG                                                            # dev_err
    assert L.mp_dispatch_rows_bulk(2, 8, 60, B.MP_BF16, P, N0, P, 16, P, N0, P, N0) == \
        B.MP_ERR_INVALID_ARG                                                            # H % 8
    L.mp_layout_and_offsets.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int64] + [ctypes.c_void_p] * 14
    assert L.mp_layout_and_offsets(2, 8, 2, 7, P, P, 16, *([P] * 13), N0) == \
        B.MP_ERR_INVALID_ARG  # E % R
    assert L.mp_layout_and_offsets(2, 8, 2, 8, P, P, 16, *([P] * 12), N0, N0) == \
        B.MP_ERR_INVALID_ARG  # workspace
    L.mp_dispatch_ll.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4 + [ctypes.c_int64] + \
        [ctypes.c_void_p] * 8
    ok = (2, 8, 2, 8, 64, B.MP_BF16, 0, P, N0, P, N0, 16, P, P, P, P, P, N0, P, N0)

    def ll(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.mp_dispatch_ll(*a)
    assert ll(a6=2) == B.MP_ERR_INVALID_ARG                                             # rank_major
    assert ll(a15=_p(FAKE + 2)) == B.MP_ERR_INVALID_ARG                                 # slot_row align
    assert ll(a16=_p(FAKE + 8)) == B.MP_ERR_INVALID_ARG                                 # recv_x align
    assert ll(a4=60) == B.MP_ERR_INVALID_ARG                                            # H % 8
    assert ll(a3=7) == B.MP_ERR_INVALID_ARG                                             # E % R
    assert ll(a5=B.MP_E4M3, a4=128) == B.MP_ERR_INVALID_ARG                             # no scales
    assert ll(a18=N0) == B.MP_ERR_INVALID_ARG                                           # dev_err
    neg = (ctypes.c_int64 * 2)(3, -1)
    assert L.mp_allgatherv_mxfp8(2, 64, neg, P, P, P, N0) == B.MP_ERR_INVALID_ARG      # size < 0
    L.mp_dispatch_noalloc.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p] * 7 + [ctypes.c_int64] + \
        [ctypes.c_void_p] * 12
    assert L.mp_dispatch_noalloc(32, 100000, 8, 256, 64, B.MP_BF16, *([P] * 7), 16,
                                 *([P] * 11), N0) == B.MP_ERR_INVALID_ARG                # > 1 MiB scratch
