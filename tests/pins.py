"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes one compiled oracle (``oracle.OracleLib``) and
raises AssertionError when the oracle disagrees with what the pages and the
mathematics fix: the hand-worked fixtures under ``tests/golden/``, brute
force over tiny inputs written with sets and sorting (not the oracle's
append loop), closed forms, special cases and library routines (torch's own
float -> bf16 rounding).  ``test_oracle_pins.py`` runs them on the oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with a planted
mistake and checks that at least one pin fails for every mistake.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from collections import Counter
from fractions import Fraction

import numpy as np
import torch

from combine_mp_layout_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits(a) -> np.ndarray:
    """float values -> bf16 bit patterns through torch's conversion (a library routine)."""
    return wl.bf16_bits(torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def _f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def load(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# bf16 conversions against torch's conversion routines
# --------------------------------------------------------------------------
def pin_bf16_rounding(orc) -> None:
    rng = np.random.default_rng(11)
    # random binary32 bit patterns over the whole finite range
    u = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    # exact ties with odd and even kept halves, values next to ties, subnormals,
    # zeros, the largest finite values and the overflow boundary
    kept = rng.integers(0, 2**16, size=4096, dtype=np.uint64).astype(np.uint32)
    ties = ((kept << 16) | 0x8000).view(np.float32)
    near = np.concatenate([((kept << 16) | 0x7fff), ((kept << 16) | 0x8001)]).view(np.float32)
    special = np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 3.4028235e38,
                        -3.4028235e38, 3.3961775e38, 1e-40, -1e-40, 1.4e-45, 2.0**-126,
                        65504.0, 0.1, 1.0 / 3.0], np.float32)
    allv = np.concatenate([f, ties[np.isfinite(ties)], near[np.isfinite(near)], special])
    got = orc.f32_to_bf16_array(allv)
    want = _bits(allv)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, "bf16 narrowing differs from torch at %r" % (allv[bad[:5]],)
    # NaN stays NaN, whatever its payload (IEEE-754: a NaN operand gives a NaN), also
    # when the payload sits only in the 16 bits that narrowing drops
    nans = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7F80FFFF, 0x7FBF0000],
                    np.uint32).view(np.float32)
    nan_bits = orc.f32_to_bf16_array(np.concatenate([np.array([np.nan, -np.nan], np.float32),
                                                     nans]))
    assert all(((int(b) & 0x7f80) == 0x7f80 and (int(b) & 0x7f) != 0) for b in nan_bits)
    # widening is exact: compare with torch's bf16 -> fp32
    b = rng.integers(0, 2**16, size=4096, dtype=np.uint64).astype(np.uint16)
    tw = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    ow = np.array([orc.bf16_to_f32(int(v)) for v in b], np.float32)
    fin = np.isfinite(tw)
    assert np.array_equal(ow[fin].view(np.uint32), tw[fin].view(np.uint32))


# --------------------------------------------------------------------------
# layout / dispatch: hand-worked fixture and brute force
# --------------------------------------------------------------------------
def pin_ep_hand_fixture(orc) -> None:
    g = load("ep_hand_r2.json")
    E, ex = g["E"], g["expect"]
    idx = np.array(g["topk_idx"], np.int32)
    w = np.array(g["topk_weights"], np.float32)
    x = _bits(g["x"])
    ntpr, ntpe, mask, st = orc.layout(idx, E)
    assert st == 0
    assert ntpr.tolist() == ex["num_tokens_per_rank"]
    assert ntpe.tolist() == ex["num_tokens_per_expert"]
    assert mask.tolist() == ex["is_token_in_rank"]
    out, st = orc.dispatch(x, idx, w, mask, E)
    assert st == 0
    for key in ("dest_offsets", "rank_prefix", "num_recv_tokens_per_expert", "send_row",
                "recv_src_rank", "recv_src_idx", "recv_topk_idx"):
        assert out[key].tolist() == ex[key], key
    assert out["recv_topk_weights"].tolist() == ex["recv_topk_weights"]
    assert np.array_equal(out["recv_x"], _bits(ex["recv_x"]))
    comb, st = orc.combine(out["recv_x"], out["send_row"])
    assert st == 0 and np.array_equal(comb, _bits(ex["combine_of_recv_x"]))
    comb, st = orc.combine(_bits(ex["y"]), out["send_row"])
    assert st == 0 and np.array_equal(comb, _bits(ex["combine_of_y"]))
    gid, st = orc.recv_topk_global(idx, E, out, 4)
    assert st == 0 and gid.tolist() == ex["recv_topk_idx_global_sentinel_4"]
    cw, st = orc.combine_weights(out["recv_topk_weights"], out["send_row"])
    assert st == 0 and cw.tolist() == ex["combined_topk_weights"]
    ll, st = orc.dispatch_ll(x, idx, E)
    assert st == 0
    assert ll["expert_offsets"].tolist() == ex["ll_expert_offsets"]
    assert ll["expert_src_offsets"].tolist() == ex["ll_expert_src_offsets"]
    assert ll["recv_src_token"].tolist() == ex["ll_recv_src_token"]
    assert ll["slot_row"].tolist() == ex["ll_slot_row"]
    assert np.array_equal(ll["recv_x"], x.reshape(-1, x.shape[-1])[ll["recv_src_token"]])
    comb, st = orc.combine_ll(ll["recv_x"], ll["slot_row"], w)
    assert st == 0 and np.array_equal(comb, _bits(ex["ll_combine_of_recv_x"]))


def brute_force_ep(topk_idx: np.ndarray, topk_weights: np.ndarray, E: int):
    """Independent formulation: experts as sets, rows as a sorted list of
    (dest, src, token) triples, counts with Counter."""
    R, N, K = topk_idx.shape
    El = E // R
    owner = {e: e // El for e in range(E)}
    triples, ntpe, ntpr, masks = [], {}, {}, {}
    for s in range(R):
        ce = Counter(int(e) for e in topk_idx[s].reshape(-1) if 0 <= e < E)
        ntpe[s] = [ce.get(e, 0) for e in range(E)]
        cr = Counter()
        for t in range(N):
            ranks = {owner[int(e)] for e in topk_idx[s, t] if 0 <= e < E}
            masks[(s, t)] = ranks
            cr.update(ranks)
            triples.extend((d, s, t) for d in ranks)
        ntpr[s] = [cr.get(d, 0) for d in range(R)]
    triples.sort()
    pos = {tr: i for i, tr in enumerate(triples)}
    return triples, pos, ntpe, ntpr, masks


def check_ep_against_brute(orc, topk_idx, topk_weights, E, x=None) -> None:
    R, N, K = topk_idx.shape
    El = E // R
    triples, pos, ntpe, ntpr, masks = brute_force_ep(topk_idx, topk_weights, E)
    o_ntpr, o_ntpe, o_mask, st = orc.layout(topk_idx, E)
    assert st == 0
    assert o_ntpe.tolist() == [ntpe[s] for s in range(R)]
    assert o_ntpr.tolist() == [ntpr[s] for s in range(R)]
    for (s, t), ranks in masks.items():
        assert {d for d in range(R) if (int(o_mask[s, t]) >> d) & 1} == ranks
    if x is None:
        x = np.arange(R * N * 8, dtype=np.uint16).reshape(R, N, 8)
    out, st = orc.dispatch(x, topk_idx, topk_weights, o_mask, E)
    assert st == 0
    T = len(triples)
    assert out["num_recv"] == T and out["dest_offsets"][R] == T
    for d in range(R):
        first = next((i for i, tr in enumerate(triples) if tr[0] >= d), T)
        assert out["dest_offsets"][d] == first
        for s in range(R):
            before = sum(1 for tr in triples if tr[0] == d and tr[1] < s)
            assert out["rank_prefix"][s, d] == before
    for i, (d, s, t) in enumerate(triples):
        assert out["recv_src_rank"][i] == s and out["recv_src_idx"][i] == t
        assert np.array_equal(out["recv_x"][i], x[s, t])
        for k in range(K):
            e = int(topk_idx[s, t, k])
            on_d = e in set(range(d * El, (d + 1) * El))
            assert out["recv_topk_idx"][i, k] == (e - d * El if on_d else -1)
            assert out["recv_topk_weights"][i, k] == (topk_weights[s, t, k] if on_d else 0.0)
    for s, t, d in itertools.product(range(R), range(N), range(R)):
        assert out["send_row"][s, t, d] == pos.get((d, s, t), -1)
    allc = Counter(int(e) for e in topk_idx.reshape(-1) if 0 <= e < E)
    assert out["num_recv_tokens_per_expert"].reshape(-1).tolist() == [allc.get(e, 0) for e in range(E)]


def pin_ep_brute_force(orc) -> None:
    rng = np.random.default_rng(3)
    for R, N, El, K in [(1, 5, 3, 2), (2, 7, 2, 3), (3, 6, 2, 4), (4, 9, 1, 3), (4, 4, 3, 12),
                        (3, 8, 4, 1)]:
        E = R * El
        idx = wl.topk_uniform(rng, R * N, E, K).reshape(R, N, K)
        # mask some entries (-1), including whole tokens
        m = rng.random(idx.shape) < 0.15
        idx = np.where(m, -1, idx).astype(np.int32)
        if N > 2:
            idx[0, 1, :] = -1
        w = rng.random(idx.shape).astype(np.float32)
        check_ep_against_brute(orc, idx, w, E)


def pin_ep_invariants(orc) -> None:
    """Invariants on a moderate random case (uniform and skewed routing)."""
    for name, over in [("tiny", {}), ("skew", dict(N=64, H=8)), ("dsv3", dict(N=32, H=8))]:
        inp = wl.make_ep(name, seed=5, **over)
        R, N, K, E = inp.R, inp.N, inp.K, inp.E
        idx = inp.topk_idx.copy()
        idx[:, ::7, 0] = -1
        ntpr, ntpe, mask, st = orc.layout(idx, E)
        assert st == 0
        masked = int((idx == -1).sum())
        assert int(ntpe.sum()) == R * N * K - masked
        pop = np.unpackbits(mask.view(np.uint8)).sum()
        assert int(ntpr.sum()) == int(pop)
        x = np.arange(R * N * 4, dtype=np.int32).reshape(R, N, 4)
        out, st = orc.dispatch(x, idx, inp.topk_weights, mask, E)
        assert st == 0
        T = out["num_recv"]
        assert int(out["dest_offsets"][-1]) == T == int(ntpr.sum())
        assert np.all(np.diff(out["dest_offsets"]) == ntpr.sum(axis=0))
        keys = list(zip(out["recv_src_rank"].tolist(), out["recv_src_idx"].tolist()))
        dest = np.searchsorted(out["dest_offsets"], np.arange(T), side="right") - 1
        trip = list(zip(dest.tolist(), *zip(*keys))) if T else []
        assert trip == sorted(trip) and len(set(trip)) == T
        assert np.array_equal(out["recv_x"], x[out["recv_src_rank"], out["recv_src_idx"]])
        # scales travel with their row: every token's scales distinct
        xs = np.arange(R * N * 3, dtype=np.float32).reshape(R, N, 3) + 0.5
        outs, st = orc.dispatch(x, idx, inp.topk_weights, mask, E, x_scales=xs)
        assert st == 0 and np.array_equal(outs["recv_scales"][:T],
                                          xs[out["recv_src_rank"], out["recv_src_idx"]])
        El = E // R
        assert out["num_recv_tokens_per_expert"].sum() == int(ntpe.sum())
        assert np.array_equal(out["num_recv_tokens_per_expert"].reshape(-1), ntpe.sum(axis=0))
        # every local topk entry of a row points at a real expert of that destination
        loc = out["recv_topk_idx"]
        assert np.all((loc == -1) | ((loc >= 0) & (loc < El)))


def pin_global_ids_and_combined_weights(orc) -> None:
    """Global ids are the local ids shifted back by d*E/R (sentinel where the local id
    is -1); combined weights of an un-modified dispatch give back each valid slot's
    weight exactly (the other destinations add +0) and +0 for masked slots."""
    inp = wl.make_ep("skew", seed=8, N=96, H=8)
    R, N, K, E = inp.R, inp.N, inp.K, inp.E
    idx = inp.topk_idx.copy()
    idx[:, ::5, 1] = -1
    _, _, mask, _ = orc.layout(idx, E)
    out, _ = orc.dispatch(np.zeros((R, N, 8), np.uint16), idx, inp.topk_weights, mask, E)
    El = E // R
    for sentinel in (E, -1, 12345):
        gid, st = orc.recv_topk_global(idx, E, out, sentinel)
        assert st == 0
        dest = np.searchsorted(out["dest_offsets"], np.arange(out["num_recv"]), side="right") - 1
        loc = out["recv_topk_idx"]
        want = np.where(loc >= 0, loc + (dest * El)[:, None], sentinel)
        assert np.array_equal(gid, want)
    cw, st = orc.combine_weights(out["recv_topk_weights"], out["send_row"])
    assert st == 0
    valid = (idx >= 0) & (idx < E)
    assert np.array_equal(cw.view(np.uint32),
                          np.where(valid, inp.topk_weights, np.float32(0)).view(np.uint32))
    # order and rounding of the sum over destinations, binary32 from +0 in ascending d:
    # the sum-order fixture's columns as the weights three destinations hold for one
    # token (slot k = column); exact binary32 results, derived by hand:
    #   (2^24 + 1) rounds to 2^24 (tie to even), minus 2^24: 0  -- both orders of col 0/1
    #   -2^24 + 2^24 + 1 = 1;  1+1+1 = 3;  0.5+0.25+0.125 = 0.875;  (+0)+(-0)+(-0) = +0;
    #   1 + 2^-8 + 0 = 1.00390625;  1 + 2^-8 + 2^-16 (exact in binary32)
    g = load("sum_order_r3.json")
    w3 = np.array(g["rows_in_rank_order"], np.float32)            # [d][k]
    send3 = np.full((3, 1, 3), -1, np.int32)
    send3[0, 0] = [0, 1, 2]
    cw, st = orc.combine_weights(w3, send3)
    want = np.array([0.0, 0.0, 1.0, 3.0, 0.875, 0.0, 1.00390625, 1.0 + 2.0**-8 + 2.0**-16],
                    np.float32)
    assert st == 0 and np.array_equal(cw[0, 0].view(np.uint32), want.view(np.uint32)), cw[0, 0]
    # a row past the rows given is flagged and skipped
    cw, st = orc.combine_weights(w3[:2], send3)
    assert st & 4 and cw[0, 0, 3] == 2.0


def pin_low_latency_layout(orc) -> None:
    """Expert-major rows against a sorted enumeration of (expert, source, token) triples;
    the weighted combine against exact sums where every step is exact."""
    rng = np.random.default_rng(17)
    for R, N, E, K in [(2, 9, 6, 3), (3, 16, 12, 4), (4, 5, 4, 4), (1, 7, 3, 2)]:
        idx = wl.topk_uniform(rng, R * N, E, K).reshape(R, N, K)
        idx[rng.random(idx.shape) < 0.2] = -1
        x = rng.integers(0, 60000, (R, N, 8)).astype(np.uint16)
        ll, st = orc.dispatch_ll(x, idx, E)
        assert st == 0
        triples = sorted((int(idx[s, t, k]), s, t, k) for s in range(R) for t in range(N)
                         for k in range(K) if idx[s, t, k] >= 0)
        assert ll["num_recv"] == len(triples) == ll["expert_offsets"][E]
        for r, (e, s, t, k) in enumerate(triples):
            assert ll["slot_row"][s, t, k] == r and ll["recv_src_token"][r] == s * N + t
            assert ll["expert_offsets"][e] <= r < ll["expert_offsets"][e + 1]
            assert np.array_equal(ll["recv_x"][r], x[s, t])
        for e in range(E):
            for s in range(R):
                before = sum(1 for tr in triples if tr[0] == e and tr[1] < s)
                assert ll["expert_src_offsets"][e, s] == before
        assert np.all(ll["slot_row"][idx < 0] == -1)
        # weights that are powers of two and small-integer rows: every product and
        # partial sum is exact, so the result is the exact weighted sum
        wts = np.exp2(-rng.integers(0, 4, idx.shape)).astype(np.float32)
        y = rng.integers(-8, 9, (ll["num_recv"], 8)).astype(np.float32)
        comb, st = orc.combine_ll(_bits(y), ll["slot_row"], wts)
        exact = np.zeros((R, N, 8))
        for s in range(R):
            for t in range(N):
                for k in range(K):
                    r = ll["slot_row"][s, t, k]
                    if r >= 0:
                        exact[s, t] += float(wts[s, t, k]) * y[r]
        assert st == 0 and np.array_equal(_f32(comb), exact.astype(np.float32))
    # receive capacity: rows are numbered as without it (the offsets count every row),
    # rows at or past it are not written, their slot_row is -1, and the call flags it
    idx = wl.topk_uniform(rng, 3 * 10, 6, 2).reshape(3, 10, 2)
    x = rng.integers(0, 60000, (3, 10, 8)).astype(np.uint16)
    full, st = orc.dispatch_ll(x, idx, 6)
    assert st == 0 and full["num_recv"] == 60
    cut, st = orc.dispatch_ll(x, idx, 6, recv_capacity=25)
    assert st & 4
    assert np.array_equal(cut["expert_offsets"], full["expert_offsets"])
    assert np.array_equal(cut["expert_src_offsets"], full["expert_src_offsets"])
    assert np.array_equal(cut["slot_row"], np.where(full["slot_row"] < 25, full["slot_row"], -1))
    assert np.array_equal(cut["recv_x"][:25], full["recv_x"][:25])


def pin_low_latency_rank_major(orc) -> None:
    """Rank-major rows against a sorted enumeration of (owner rank, source, token, slot)
    tuples; the same rows as the expert-major layout, regrouped."""
    rng = np.random.default_rng(19)
    for R, N, E, K in [(2, 9, 6, 3), (3, 16, 12, 4), (4, 5, 4, 4), (1, 7, 3, 2)]:
        idx = wl.topk_uniform(rng, R * N, E, K).reshape(R, N, K)
        idx[rng.random(idx.shape) < 0.2] = -1
        x = rng.integers(0, 60000, (R, N, 8)).astype(np.uint16)
        rm, st = orc.dispatch_ll_rank_major(x, idx, E)
        assert st == 0
        El = E // R
        tuples = sorted((int(idx[s, t, k]) // El, s, t, k) for s in range(R) for t in range(N)
                        for k in range(K) if idx[s, t, k] >= 0)
        assert rm["num_recv"] == len(tuples) == rm["dest_offsets"][R]
        for r, (d, s, t, k) in enumerate(tuples):
            assert rm["slot_row"][s, t, k] == r and rm["recv_src_token"][r] == s * N + t
            assert rm["dest_offsets"][d] <= r < rm["dest_offsets"][d + 1]
            assert np.array_equal(rm["recv_x"][r], x[s, t])
        for d in range(R):
            for s in range(R):
                before = sum(1 for tu in tuples if tu[0] == d and tu[1] < s)
                assert rm["dest_src_offsets"][d, s] == before
        assert np.all(rm["slot_row"][idx < 0] == -1)
        # the same (token, slot) rows as the expert-major layout, and per destination the
        # expert-major blocks of its experts hold exactly as many rows
        em, st = orc.dispatch_ll(x, idx, E)
        assert st == 0 and np.array_equal(rm["slot_row"] >= 0, em["slot_row"] >= 0)
        for d in range(R):
            assert (rm["dest_offsets"][d + 1] - rm["dest_offsets"][d]
                    == em["expert_offsets"][(d + 1) * El] - em["expert_offsets"][d * El])
    # a too-small capacity keeps the first rows and flags the rest
    idx = wl.topk_uniform(rng, 2 * 6, 4, 2).reshape(2, 6, 2)
    x = rng.integers(0, 60000, (2, 6, 8)).astype(np.uint16)
    full, _ = orc.dispatch_ll_rank_major(x, idx, 4)
    cut, st = orc.dispatch_ll_rank_major(x, idx, 4, recv_capacity=10)
    assert st == 4 and np.array_equal(cut["recv_src_token"], full["recv_src_token"][:10])
    assert np.array_equal(cut["slot_row"], np.where(full["slot_row"] < 10, full["slot_row"], -1))

def pin_ep_special_cases(orc) -> None:
    rng = np.random.default_rng(9)
    # R = 1: dispatch is the identity on tokens with an expert; combine gives them back
    idx = wl.topk_uniform(rng, 10, 4, 2).reshape(1, 10, 2)
    idx[0, 3] = -1
    w = rng.random(idx.shape).astype(np.float32)
    x = _bits(rng.standard_normal((1, 10, 8)))
    _, _, mask, _ = orc.layout(idx, 4)
    out, st = orc.dispatch(x, idx, w, mask, 4)
    keep = [t for t in range(10) if t != 3]
    assert st == 0 and np.array_equal(out["recv_x"], x[0, keep])
    comb, _ = orc.combine(out["recv_x"], out["send_row"])
    assert np.array_equal(comb[0, keep], x[0, keep]) and not comb[0, 3].any()
    # K = E: every token goes to every rank, R*N*R rows
    R, N, E = 3, 4, 6
    idx = np.tile(np.arange(E, dtype=np.int32), (R, N, 1))
    _, ntpe, mask, _ = orc.layout(idx, E)
    assert np.all(mask == (1 << R) - 1) and np.all(ntpe == N)
    out, _ = orc.dispatch(np.zeros((R, N, 8), np.uint16), idx, np.ones(idx.shape, np.float32),
                          mask, E)
    assert out["num_recv"] == R * N * R
    # everything masked: no rows, zero counts, combine gives +0 rows
    idx = np.full((2, 5, 3), -1, np.int32)
    ntpr, ntpe, mask, st = orc.layout(idx, 4)
    assert st == 0 and not ntpr.any() and not ntpe.any() and not mask.any()
    out, st = orc.dispatch(np.ones((2, 5, 8), np.uint16), idx, np.ones(idx.shape, np.float32),
                           mask, 4)
    assert st == 0 and out["num_recv"] == 0 and np.all(out["send_row"] == -1)
    comb, _ = orc.combine(np.zeros((1, 8), np.uint16), out["send_row"])
    assert not comb.any()
    # bad expert ids are flagged and ignored
    idx = np.array([[[0, 9], [-3, 1]]], np.int32)
    ntpr, ntpe, mask, st = orc.layout(idx, 2)
    assert st & 8 and mask.tolist() == [[1, 1]] and ntpe.tolist() == [[1, 1]]
    # receive capacity: rows past it are not written and their send_row is -1
    idx = np.array([[[0], [1], [0]], [[1], [0], [1]]], np.int32)
    _, _, mask, _ = orc.layout(idx, 2)
    x = np.arange(2 * 3 * 8, dtype=np.uint16).reshape(2, 3, 8)
    out, st = orc.dispatch(x, idx, np.ones(idx.shape, np.float32), mask, 2, recv_capacity=4)
    assert st & 4 and out["num_recv"] == 6
    assert int((out["send_row"] >= 0).sum()) == 4 and out["send_row"].max() == 3
    # ... the capacity only truncates: the offset tables still describe every row (the
    # exact need is dest_offsets[R]), rows below it are those of an unlimited run
    full, st = orc.dispatch(x, idx, np.ones(idx.shape, np.float32), mask, 2)
    assert st == 0 and full["dest_offsets"].tolist() == [0, 3, 6]
    assert np.array_equal(out["dest_offsets"], full["dest_offsets"])
    assert np.array_equal(out["rank_prefix"], full["rank_prefix"])
    assert np.array_equal(out["send_row"], np.where(full["send_row"] < 4, full["send_row"], -1))
    assert np.array_equal(out["recv_x"][:4], full["recv_x"][:4])
    # combine: a send_row entry past the rows given is flagged and skipped
    y = _bits(np.arange(1, 7, dtype=np.float32)[:, None].repeat(8, axis=1))
    comb, st = orc.combine(y[:4], full["send_row"])
    assert st & 4
    got = _f32(comb)[..., 0]
    for s_, t_ in itertools.product(range(2), range(3)):
        r = [v for v in full["send_row"][s_, t_] if 0 <= v < 4]
        assert got[s_, t_] == sum(float(r_ + 1) for r_ in r)


# --------------------------------------------------------------------------
# combine / reduce-scatterv sums
# --------------------------------------------------------------------------
def pin_sum_order_fixture(orc) -> None:
    g = load("sum_order_r3.json")
    rows = _bits(g["rows_in_rank_order"])          # [3][8]
    want = np.array([int(h, 16) for h in g["expect_bf16_bits"]], np.uint16)
    # as a combine: one token of source rank 0 sent to ranks 0, 1, 2 (rows 0, 1, 2)
    send_row = np.full((3, 1, 3), -1, np.int32)
    send_row[0, 0] = [0, 1, 2]
    out, st = orc.combine(rows, send_row)
    assert st == 0 and np.array_equal(out[0, 0], want), out[0, 0]
    assert not out[1:].any()
    # as a reduce-scatterv: rank q's one-row input is row q; the row is rank 1's shard
    out, st = orc.reducescatterv(rows.reshape(3, 1, 8), [0, 1, 0])
    assert st == 0 and np.array_equal(out[0], want)


def pin_low_latency_combine_closed_forms(orc) -> None:
    """The weighted low-latency combine.  With unit weights every product is exact, so it
    is the plain sum of the hand-worked sum-order fixture, slots taken in ascending k (a
    masked slot contributes nothing).  Each product is rounded to binary32 before it is
    added: w*y with w = 1 + 2^-20 and y = 1 + 2^-7 is 1 + 2^-7 + 2^-20 + 2^-27, which
    rounds to 1 + 2^-7 + 2^-20, so adding the product of -w and y cancels it to +0,
    where a fused multiply-add would leave -2^-27."""
    g = load("sum_order_r3.json")
    rows = _bits(g["rows_in_rank_order"])          # [3][8]
    want = np.array([int(h, 16) for h in g["expect_bf16_bits"]], np.uint16)
    out, st = orc.combine_ll(rows, np.array([[[0, 1, 2]]], np.int32),
                             np.ones((1, 1, 3), np.float32))
    assert st == 0 and np.array_equal(out[0, 0], want), out[0, 0]
    out, st = orc.combine_ll(rows, np.array([[[0, -1, 1, 2]]], np.int32),
                             np.ones((1, 1, 4), np.float32))
    assert st == 0 and np.array_equal(out[0, 0], want), out[0, 0]
    y = _bits(np.full((2, 8), 1.0 + 2.0**-7, np.float32))
    w = np.array([[[1.0 + 2.0**-20, -(1.0 + 2.0**-20)]]], np.float32)
    out, st = orc.combine_ll(y, np.array([[[0, 1]]], np.int32), w)
    assert st == 0 and not out.any(), [hex(int(b)) for b in out[0, 0]]


def pin_combine_closed_forms(orc) -> None:
    rng = np.random.default_rng(21)
    inp = wl.make_ep("dsv3", seed=2, N=48, H=64)
    R, N, E = inp.R, inp.N, inp.E
    idx = inp.topk_idx.copy()
    idx[1, 5] = -1
    _, _, mask, _ = orc.layout(idx, E)
    x = wl.bf16_bits(inp.x)
    out, _ = orc.dispatch(x, idx, inp.topk_weights, mask, E)
    # combine of an un-modified dispatch is bf16(c * x), c = number of destination
    # ranks (c*x is exact in fp32 for bf16 x and c <= 32; one rounding by torch)
    c = np.unpackbits(mask.view(np.uint8).reshape(R, N, 4), axis=-1).sum(-1).astype(np.float32)
    want = _bits(_f32(x) * c[..., None])
    want[c == 0] = 0  # no destination: the +0.0 start value, not 0 * x (which may be -0)
    comb, st = orc.combine(out["recv_x"], out["send_row"])
    assert st == 0 and np.array_equal(comb, want)
    # small-integer rows: every fp32 partial sum is exact, so the result is the
    # exact integer sum (|sum| <= 8*16 fits bf16's 8 significant bits)
    T = out["num_recv"]
    yi = rng.integers(-16, 17, size=(T, 64)).astype(np.float32)
    comb, _ = orc.combine(_bits(yi), out["send_row"])
    exact = np.zeros((R, N, 64), np.float64)
    for s, t, d in itertools.product(range(R), range(N), range(R)):
        r = out["send_row"][s, t, d]
        if r >= 0:
            exact[s, t] += yi[r]
    assert np.array_equal(_f32(comb), exact.astype(np.float32))
    # random rows: within the fp32 recursive-summation bound of the exact sum
    # plus half a bf16 ulp of the final rounding
    yr = rng.standard_normal((T, 64)).astype(np.float32)
    yb = _bits(yr)
    yv = _f32(yb).astype(np.float64)
    comb, _ = orc.combine(yb, out["send_row"])
    got = _f32(comb).astype(np.float64)
    for s, t in itertools.product(range(R), range(N)):
        rows = [r for r in out["send_row"][s, t] if r >= 0]
        if not rows:
            assert not comb[s, t].any()
            continue
        for h in range(0, 64, 7):
            vals = [Fraction(float(yv[r, h])) for r in rows]
            ex = float(sum(vals, Fraction(0)))
            absum = float(sum(abs(v) for v in vals))
            bound = (len(rows) - 1) * 2.0**-24 * absum * 1.01 + 2.0**-8 * abs(ex) * 1.01 + 1e-30
            assert abs(got[s, t, h] - ex) <= bound, (s, t, h, got[s, t, h], ex)


def pin_rsv_agv(orc) -> None:
    rng = np.random.default_rng(33)
    R, H = 8, 16
    sizes = [3, 0, 5, 1, 0, 2, 4, 1]
    S = sum(sizes)
    shard = _bits(rng.standard_normal((S, H)))
    # all-gatherv: every logical rank's output is the shards concatenated in rank order
    ag, st = orc.allgatherv(shard, sizes, R)
    assert st == 0 and ag.shape == (R, S, H)
    off = np.concatenate([[0], np.cumsum(sizes)])
    for q, r in itertools.product(range(R), range(R)):
        assert np.array_equal(ag[q, off[r]:off[r + 1]], shard[off[r]:off[r + 1]])
    # round trip: reduce-scatterv of the gathered copies is bf16(R * shard), exact for R = 8
    rs, st = orc.reducescatterv(ag, sizes)
    assert st == 0 and np.array_equal(rs, _bits(_f32(shard) * np.float32(R)))
    # small integers: exact sums
    xi = rng.integers(-16, 17, size=(R, S, H)).astype(np.float32)
    rs, _ = orc.reducescatterv(_bits(xi), sizes)
    assert np.array_equal(_f32(rs), xi.sum(0, dtype=np.float64).astype(np.float32))
    # random: within the summation bound
    xr = _f32(_bits(rng.standard_normal((R, S, H)))).astype(np.float64)
    rs, _ = orc.reducescatterv(_bits(xr), sizes)
    ex = np.array([[math.fsum(xr[:, i, h]) for h in range(H)] for i in range(S)])
    bound = (R - 1) * 2.0**-24 * np.abs(xr).sum(0) * 1.01 + 2.0**-8 * np.abs(ex) * 1.01 + 1e-30
    assert np.all(np.abs(_f32(rs) - ex) <= bound)
    # empty shards everywhere: nothing to do
    rs, st = orc.reducescatterv(np.zeros((3, 0, 8), np.uint16), [0, 0, 0])
    assert st == 0 and rs.shape == (0, 8)


NONFINITE_CASES = [  # (addends in ascending rank order, expected bf16 bits; None = a NaN)
    ([np.inf, 1.0], 0x7F80), ([1.0, -np.inf], 0xFF80), ([np.inf, np.inf], 0x7F80),
    ([np.inf, -np.inf], None), ([np.nan, 1.0], None), ([1.0, 2.0, np.nan], None),
    ([3.3895314e38, 3.3895314e38], 0x7F80),      # binary32 overflow: +Inf
    ([-3.3895314e38, -3.3895314e38], 0xFF80),
    ([3.3895314e38, 2.0**118], 0x7F7F),          # 0x7F7F4000: below the midpoint
    ([3.3895314e38, 2.0**118, 2.0**117], 0x7F7F),  # 0x7F7F6000: still below
    ([3.3895314e38, 2.0**118, 2.0**118], 0x7F80),  # 0x7F7F8000: a tie, odd kept half: up
    ([-0.0, -0.0], 0x0000),                      # +0.0 start: (+0) + (-0) = +0
    ([-0.0], 0x0000),
    ([2.0**-126, -(2.0**-126)], 0x0000),         # exact cancellation to +0
]


def is_bf16_nan(bits) -> bool:
    b = int(bits)
    return (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


def pin_nonfinite_sums(orc) -> None:
    """IEEE-754 closed forms for the combine's and the reduce-scatterv's sums: binary32
    adds from +0.0 in rank order, then one round-to-nearest-even to bf16.  An infinity
    survives, Inf + -Inf and NaN give NaN, a binary32 overflow gives Inf, and a sum
    above bf16's largest finite value (0x7F7F = (2 - 2^-7) * 2^127, its ulp 2^120)
    rounds up only from the midpoint 0x7F7F8000 on."""
    H = 8
    for addends, want in NONFINITE_CASES:
        n = len(addends)
        rows = _bits(np.repeat(np.array(addends, np.float32)[:, None], H, axis=1))
        a32 = np.array(addends, np.float32)
        fin = ~np.isnan(a32)  # every addend is a bf16 value (NaNs: any NaN)
        assert np.array_equal(_f32(rows)[fin, 0].view(np.uint32), a32[fin].view(np.uint32))
        assert np.isnan(_f32(rows)[~fin, 0]).all(), addends
        send_row = np.full((n, 1, n), -1, np.int32)
        send_row[0, 0] = np.arange(n)
        comb, st = orc.combine(rows, send_row)
        sizes = [0] * n
        sizes[n - 1] = 1
        rs, st2 = orc.reducescatterv(rows.reshape(n, 1, H), sizes)
        assert st == 0 and st2 == 0
        for got in (comb[0, 0], rs[0]):
            if want is None:
                assert all(is_bf16_nan(b) for b in got), (addends, got)
            else:
                assert all(int(b) == want for b in got), (addends, [hex(int(b)) for b in got])


# --------------------------------------------------------------------------
# FP8 E4M3 narrowing and per-128-channel block quantisation
# --------------------------------------------------------------------------
def _torch_e4m3(vals: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def pin_e4m3_conversions(orc) -> None:
    rng = np.random.default_rng(41)
    # every finite code decodes like torch's float8_e4m3fn
    codes = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], np.uint8)
    tdec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    odec = np.array([orc.e4m3_to_f32(int(c)) for c in codes], np.float32)
    assert np.array_equal(odec, tdec)
    # narrowing: random binary32 values inside the finite range, every code value,
    # every midpoint between neighbouring codes (ties) and values just either side
    mags = np.sort(np.unique(np.abs(tdec)))
    mids = (mags[:-1].astype(np.float64) + mags[1:]) / 2
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1000))])
    rnd = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000))).astype(np.float32)
    allv = np.concatenate([mags, mids.astype(np.float32), near, rnd]).astype(np.float32)
    allv = allv[np.abs(allv) <= 448]
    allv = np.concatenate([allv, -allv])
    ours = np.array([orc.f32_to_e4m3(float(v)) for v in allv], np.uint8)
    theirs = _torch_e4m3(allv)
    bad = np.nonzero(ours != theirs)[0]
    assert bad.size == 0, allv[bad[:5]]
    # saturation to +-448 above the range (satfinite), NaN stays NaN
    for v in (449.0, 464.0, 500.0, 1e6, float("inf")):
        assert orc.f32_to_e4m3(v) == 0x7e and orc.f32_to_e4m3(-v) == 0xfe
    assert orc.f32_to_e4m3(float("nan")) & 0x7f == 0x7f


def pin_block_quantisation(orc) -> None:
    rng = np.random.default_rng(43)
    x = (rng.standard_normal((40, 512)) * np.exp2(rng.integers(-6, 6, (40, 1)))).astype(np.float32)
    x[3, :128] = 0.0                     # an all-zero block: scale 1, codes 0
    x[4, 128:256] = 2.5                  # a constant block: every code is 448
    x[5, 256:384] = -x[5, 256:384]
    xb = _bits(x)
    xf = _f32(xb).astype(np.float64)
    q, sc, st = orc.quantize_e4m3(xb)
    assert st == 0 and q.shape == x.shape and sc.shape == (40, 4)
    blocks = xf.reshape(40, 4, 128)
    amax = np.abs(blocks).max(-1)
    want_scale = np.where(amax > 0, (amax.astype(np.float32) / np.float32(448)), 1.0)
    assert np.array_equal(sc, want_scale.astype(np.float32))
    assert sc[3, 0] == 1.0 and not q[3, :128].any()
    assert np.all(q[4, 128:256] == 0x7e)
    # the largest element of every non-zero block lands on the largest code
    qb = q.reshape(40, 4, 128)
    for t, b in zip(*np.nonzero(amax > 0)):
        j = int(np.abs(blocks[t, b]).argmax())
        assert qb[t, b, j] & 0x7f == 0x7e
    # dequantised values are within half an e4m3 step of x (relative 2^-4 for
    # normals, 2^-10 * scale below the normal range), the sign is kept
    deq = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    deq = (deq.reshape(40, 4, 128) * sc[..., None]).reshape(40, 512)
    tol = np.maximum(np.abs(xf) * 2.0**-4, np.repeat(sc, 128, axis=1) * 2.0**-10) * 1.0001
    assert np.all(np.abs(deq - xf) <= tol)
    assert np.all((deq == 0) | (np.sign(deq) == np.sign(xf)))
    # every code exactly: the binary32 quotient x / scale correctly rounded (numpy's
    # float32 division is IEEE-754's), narrowed by torch's e4m3 cast with the
    # satfinite clamp at +-448 of the reading
    x32 = _f32(xb).reshape(40, 4, 128)
    quo = np.clip(x32 / sc[..., None], np.float32(-448), np.float32(448))
    assert np.array_equal(q, _torch_e4m3(quo.reshape(40, 512)))
    # blocks whose elements sit where x * RN(1 / scale) and RN(x / scale) narrow to
    # different codes: they pin the division itself (a reciprocal taken first moves
    # these across an e4m3 rounding boundary)
    bf16_pos = (np.arange(1, 0x7f80, dtype=np.uint32) << 16).view(np.float32)
    rows = []
    for a_bits in (0x4118, 0x3fd0, 0x4944, 0x4b44, 0x4c52, 0x42d2):
        amax_b = np.float32((np.uint32(a_bits) << 16).view(np.float32))
        scale = np.float32(amax_b / np.float32(448))
        cand = bf16_pos[bf16_pos < amax_b]
        by_div = _torch_e4m3(np.clip(cand / scale, 0, 448))
        by_rcp = _torch_e4m3(np.clip(cand * (np.float32(1) / scale), 0, 448))
        hard = cand[by_div != by_rcp][:63]
        assert hard.size > 0
        blk = np.zeros(128, np.float32)
        blk[0] = amax_b
        blk[1:1 + hard.size] = hard
        blk[64:64 + hard.size] = -hard
        rows.append(blk)
    xh = _bits(np.stack(rows))
    qh, sch, st = orc.quantize_e4m3(xh)
    assert st == 0
    quo = np.clip(_f32(xh) / sch, np.float32(-448), np.float32(448))
    assert np.array_equal(qh, _torch_e4m3(quo))


def pin_mxfp8_quantisation(orc) -> None:
    """Scale codes against numpy's frexp (an independent exponent extraction); the
    block maximum lands in the top binade of e4m3; decoded values within half an e4m3
    step of x; all-zero blocks code 0; tiny non-zero blocks kept at code 0."""
    rng = np.random.default_rng(47)
    x = (rng.standard_normal((30, 256)) * np.exp2(rng.integers(-20, 20, (30, 8)).repeat(32, 1)))
    x = x.astype(np.float32)
    x[2, :32] = 0.0                                   # all-zero block
    x[3, 32:64] = np.float32(2.0**-130) * rng.integers(1, 8, 32)  # tiny non-zero block
    xb = _bits(x)
    xf = _f32(xb).astype(np.float64)
    q, codes, st = orc.quantize_mxfp8(xb)
    assert st == 0 and codes.shape == (30, 8)
    amax = np.abs(xf.reshape(30, 8, 32)).max(-1)
    mant, ex = np.frexp(amax)                         # amax = mant * 2^ex, mant in [0.5, 1)
    want = np.where(amax > 0, np.clip(ex - 1 - 8 + 127, 0, 254), 0)
    assert np.array_equal(codes.astype(np.int64), want)
    assert codes[2, 0] == 0 and not q[2, :32].any()
    assert codes[3, 1] == 0 and q[3, 32:64].any()
    deq = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    X = np.exp2(codes.astype(np.float64) - 127)
    deq = (deq.reshape(30, 8, 32) * X[..., None]).reshape(30, 256)
    tol = np.maximum(np.abs(xf) * 2.0**-4, np.repeat(X, 32, axis=1) * 2.0**-10) * 1.0001
    normal = codes.repeat(32, 1) > 0
    Xe = np.repeat(X, 32, axis=1)
    sat = np.abs(xf) >= 448 * Xe   # x / X above E4M3's largest finite value: clamped
    assert np.all(np.abs(deq - xf)[normal & ~sat] <= tol[normal & ~sat])
    assert np.all(np.abs(deq)[sat] == (448 * Xe)[sat])
    qb = q.reshape(30, 8, 32)
    for t, b in zip(*np.nonzero((amax > 0) & (codes > 0))):
        j = int(np.abs(xf.reshape(30, 8, 32)[t, b]).argmax())
        mag = torch.tensor([int(qb[t, b, j]) & 0x7f], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        assert 256.0 <= mag <= 448.0


def _e2m1_by_binade(v: np.ndarray) -> np.ndarray:
    """E2M1 narrowing written independently of the oracle: scale each binade so that
    the format's step becomes 1, round with numpy's round-half-to-even, scale back,
    saturate at 6; the code is the position of the magnitude in the value grid."""
    a = np.abs(v.astype(np.float64))
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    r = np.minimum(np.round(a / step) * step, 6.0)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    code = np.searchsorted(grid, r).astype(np.uint8)
    assert np.array_equal(grid[code], r)
    return code | np.where(np.signbit(v), 8, 0).astype(np.uint8)


def pin_mxfp4_quantisation(orc) -> None:
    """E2M1 decoding against the bit layout (bias 1); narrowing against a binade-scaled
    numpy round-half-to-even; scale codes against numpy's frexp; nibble order; decoded
    values within half an E2M1 step of x / X; zero and tiny blocks."""
    for c in range(16):  # sign, 2 exponent bits (bias 1), 1 mantissa bit
        e, m = (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert orc.e2m1_to_f32(c) == (-mag if c & 8 else mag)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(53)
    vals = np.concatenate([grid, mids, np.nextafter(mids, 0), np.nextafter(mids, 10), [6.5, 7.0, 8.0, 1e30],
                           rng.standard_normal(4000) * 3]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    ours = np.array([orc.f32_to_e2m1(float(v)) for v in vals], np.uint8)
    assert np.array_equal(ours, _e2m1_by_binade(vals))
    x = (rng.standard_normal((24, 128)) * np.exp2(rng.integers(-20, 20, (24, 4)).repeat(32, 1)))
    x = x.astype(np.float32)
    x[2, :32] = 0.0                                            # all-zero block
    x[3, 32:64] = np.float32(2.0**-130) * rng.integers(1, 8, 32)  # tiny non-zero block
    x[4, 64:96] = np.tile([1.0, 6.0], 16) * 2.0**5             # even channels 1*X, odd 6*X
    xb = _bits(x)
    xf = _f32(xb).astype(np.float64)
    q, codes, st = orc.quantize_mxfp4(xb)
    assert st == 0 and q.shape == (24, 64) and codes.shape == (24, 4)
    amax = np.abs(xf.reshape(24, 4, 32)).max(-1)
    _, ex = np.frexp(amax)
    want = np.where(amax > 0, np.clip(ex - 1 - 2 + 127, 0, 254), 0)
    assert np.array_equal(codes.astype(np.int64), want)
    assert codes[2, 0] == 0 and not q[2, :16].any()
    assert codes[3, 1] == 0 and q[3, 16:32].any()
    # amax 6 * 2^5 = 192: floor(log2) 7, code 127 + 7 - 2, X = 2^5; 1*X -> code 2, 6*X -> 7
    assert codes[4, 2] == 127 + 5 and np.all(q[4, 32:48] == 0x72)
    lo, hi = q & 0x0F, q >> 4
    el = np.stack([lo, hi], axis=-1).reshape(24, 128)
    sign = np.where(el & 8, -1.0, 1.0)
    deq = sign * grid[el & 7] * np.repeat(np.exp2(codes.astype(np.float64) - 127), 32, axis=1)
    Xe = np.repeat(np.exp2(codes.astype(np.float64) - 127), 32, axis=1)
    sat = np.abs(xf) >= 6 * Xe
    tol = np.maximum(np.abs(xf) / 4, 0.25 * Xe) * 1.0001
    assert np.all(np.abs(deq - xf)[~sat] <= tol[~sat])
    assert np.all(np.abs(deq)[sat] == (6 * Xe)[sat])
    assert np.all(np.signbit(deq) == np.signbit(xf))


ALL_PINS = [pin_nonfinite_sums, pin_low_latency_combine_closed_forms, pin_bf16_rounding, pin_ep_hand_fixture, pin_ep_brute_force, pin_ep_invariants,
            pin_ep_special_cases, pin_sum_order_fixture, pin_combine_closed_forms, pin_rsv_agv,
            pin_e4m3_conversions, pin_block_quantisation, pin_global_ids_and_combined_weights,
            pin_low_latency_layout, pin_mxfp8_quantisation, pin_mxfp4_quantisation,
            pin_low_latency_rank_major]
