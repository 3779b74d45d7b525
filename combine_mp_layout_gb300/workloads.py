"""Seeded synthetic inputs for the MoE dispatch/combine and the variable-size
reduce-scatterv / all-gatherv workloads.

This module only draws random inputs; it holds none of the method's
arithmetic (no layout, offsets, copies or sums), so the CUDA path and the
CPU oracle can both be fed from it without sharing any of the computation.

Input recipe (the same for tests, the smoke check and the benchmark):
  * routing "uniform": each token picks K distinct experts out of E, the
    first K entries of a uniformly random permutation (column order kept);
  * routing "zipf": expert e has popularity (e+1)^-s (no shuffle, so the
    low experts -- and rank 0 -- are hot); the K experts are drawn one after
    another without replacement, renormalising each time.  Drawn here with
    the equivalent Gumbel-top-K construction (the order of the K largest
    log(p_e) + Gumbel keys has exactly that successive-sampling law);
  * topk_weights: softmax over the token's K standard-normal logits, fp32;
  * x: standard normal, rounded to bf16 (or cast to fp8 e4m3 with one fp32
    scale per 128 channels drawn from U[0.5, 2));
  * reduce-scatterv / all-gatherv: per-rank row counts uniform in
    [0, max_rows], inputs standard normal bf16.
Seed 0 everywhere unless a test asks for another one.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# Workloads, named by what they are.  "tiny" is the small case the oracle
# finishes instantly; "dsv3" is the DeepSeek-V3-shaped case the benchmark
# times; the others are parity cases.
CONFIGS = {
    "tiny": dict(kind="ep", R=2, N=64, H=128, E=8, K=2, routing="uniform", dtype="bf16"),
    "dsv3": dict(kind="ep", R=8, N=4096, H=7168, E=256, K=8, routing="uniform", dtype="bf16"),
    "skew": dict(kind="ep", R=16, N=2048, H=4096, E=64, K=6, routing="zipf", zipf_s=1.2,
                 dtype="bf16"),
    "fp8": dict(kind="ep", R=8, N=8192, H=7168, E=256, K=8, routing="uniform", dtype="e4m3"),
    "rsv": dict(kind="rsv", R=8, H=4096, max_rows=16384),
}

SCALE_BLOCK = 128  # channels per fp32 scale in the e4m3 payload


def topk_uniform(rng: np.random.Generator, T: int, E: int, K: int) -> np.ndarray:
    """[T][K] int32: first K entries of a uniform random permutation of range(E)."""
    if T == 0:
        return np.zeros((0, K), np.int32)
    keys = rng.random((T, E))
    part = np.argpartition(keys, K - 1, axis=1)[:, :K] if K < E else np.tile(np.arange(E), (T, 1))
    order = np.argsort(np.take_along_axis(keys, part, axis=1), axis=1)
    return np.take_along_axis(part, order, axis=1).astype(np.int32)


def topk_zipf(rng: np.random.Generator, T: int, E: int, K: int, s: float) -> np.ndarray:
    """[T][K] int32: K experts drawn in turn without replacement, p_e ~ (e+1)^-s."""
    if T == 0:
        return np.zeros((0, K), np.int32)
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    g = -np.log(-np.log(rng.random((T, E))))  # Gumbel(0,1)
    keys = logp[None, :] + g
    part = np.argpartition(-keys, K - 1, axis=1)[:, :K] if K < E else np.tile(np.arange(E), (T, 1))
    order = np.argsort(-np.take_along_axis(keys, part, axis=1), axis=1)
    return np.take_along_axis(part, order, axis=1).astype(np.int32)


def softmax_weights(rng: np.random.Generator, R: int, N: int, K: int) -> np.ndarray:
    logits = rng.standard_normal((R, N, K), dtype=np.float32)
    m = logits.max(axis=-1, keepdims=True) if N else logits
    e = np.exp(logits - m, dtype=np.float32)
    return (e / e.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor's bit patterns as a uint16 numpy array (CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


@dataclass
class EPInputs:
    R: int
    N: int
    H: int
    E: int
    K: int
    dtype: str
    topk_idx: np.ndarray          # int32 [R][N][K], -1 = masked
    topk_weights: np.ndarray      # fp32  [R][N][K]
    x: torch.Tensor               # bf16 [R][N][H] or float8_e4m3fn [R][N][H] (CPU)
    x_scales: torch.Tensor | None = None  # fp32 [R][N][H/128] for e4m3
    meta: dict = field(default_factory=dict)

    @property
    def row_bytes(self) -> int:
        return self.H * (2 if self.dtype == "bf16" else 1)


def _torch_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(0x5EED0000 + seed)
    return g


def make_ep(name_or_cfg, seed: int = 0, **overrides) -> EPInputs:
    cfg = dict(CONFIGS[name_or_cfg]) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    cfg.update(overrides)
    R, N, H, E, K = cfg["R"], cfg["N"], cfg["H"], cfg["E"], cfg["K"]
    rng = np.random.default_rng(seed)
    if cfg.get("routing", "uniform") == "zipf":
        idx = topk_zipf(rng, R * N, E, K, cfg.get("zipf_s", 1.2))
    else:
        idx = topk_uniform(rng, R * N, E, K)
    topk_idx = idx.reshape(R, N, K)
    w = softmax_weights(rng, R, N, K)
    g = _torch_gen(seed)
    dtype = cfg.get("dtype", "bf16")
    if dtype == "bf16":
        x = torch.randn((R, N, H), generator=g, dtype=torch.float32).to(torch.bfloat16)
        xs = None
    else:
        x = torch.randn((R, N, H), generator=g, dtype=torch.float32).to(torch.float8_e4m3fn)
        xs = torch.rand((R, N, H // SCALE_BLOCK), generator=g, dtype=torch.float32) * 1.5 + 0.5
    return EPInputs(R, N, H, E, K, dtype, topk_idx, w, x, xs, meta=dict(cfg, seed=seed))


def random_bf16(shape, seed: int) -> torch.Tensor:
    """Standard-normal bf16 tensor on the CPU (e.g. synthetic expert outputs)."""
    return torch.randn(tuple(shape), generator=_torch_gen(seed + 7919),
                       dtype=torch.float32).to(torch.bfloat16)


@dataclass
class RSVInputs:
    R: int
    H: int
    sizes: np.ndarray      # int64 [R]
    x: torch.Tensor        # bf16 [R][S][H]: logical rank q's reduce-scatterv input
    shards: torch.Tensor   # bf16 [S][H]: rank r's all-gatherv shard at rows off_r..

    @property
    def S(self) -> int:
        return int(self.sizes.sum())


def make_rsv(name_or_cfg="rsv", seed: int = 0, **overrides) -> RSVInputs:
    cfg = dict(CONFIGS[name_or_cfg]) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    cfg.update(overrides)
    R, H = cfg["R"], cfg["H"]
    rng = np.random.default_rng(seed)
    if "sizes" in cfg:
        sizes = np.asarray(cfg["sizes"], np.int64)
    else:
        sizes = rng.integers(0, cfg["max_rows"] + 1, size=R).astype(np.int64)
    S = int(sizes.sum())
    g = _torch_gen(seed)
    x = torch.randn((R, S, H), generator=g, dtype=torch.float32).to(torch.bfloat16)
    shards = torch.randn((S, H), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return RSVInputs(R, H, sizes, x, shards)


def random_bf16_rows(rows: int, H: int, seed: int, chunk: int = 32768) -> torch.Tensor:
    """[rows][H] standard-normal bf16 (CPU), every row drawn independently; made in
    chunks of rows (each with its own seed) so that full-size expert outputs need no
    full-size fp32 temporary."""
    out = torch.empty((rows, H), dtype=torch.bfloat16)
    for c, r0 in enumerate(range(0, rows, chunk)):
        r1 = min(rows, r0 + chunk)
        out[r0:r1] = torch.randn((r1 - r0, H), generator=_torch_gen(seed * 100003 + c + 1),
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def gathered_bf16(rows: int, H: int, seed: int, table_rows: int = 1024) -> torch.Tensor:
    """[rows][H] bf16 synthetic expert outputs made cheaply at large sizes: each row is
    a row of a standard-normal table picked uniformly at random (CPU)."""
    table = random_bf16((table_rows, H), seed)
    pick = torch.from_numpy(np.random.default_rng(seed + 17).integers(0, table_rows, rows))
    return table.index_select(0, pick)
