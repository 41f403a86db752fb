"""Seeded synthetic workloads for the NABLA mask builder and sparse attention.

This module holds only shapes and random draws. It contains none of the
method's arithmetic (no pooling, no softmax, no thresholding, no attention),
so both the CUDA path and the fp64 oracle can be fed from it without sharing
any computation.

Inputs stand in for video-DiT latents: the NABLA pages measure on Wan 2.1 /
a 2B DiT, whose weights and prompts are not available, so q/k/v are drawn from
a block-structured Gaussian whose block grid has the (T, H, W) shape of a
480p- or 720p-like latent ("NABLA: Neighborhood Adaptive Block-Level
Attention", Technical Summary, Experimental Results).

Generator (same for every configuration, seed 0 unless stated):
  * numpy SeedSequence(seed) spawns five streams, in this order: m_q, n_q,
    m_k, n_k, v; each token tensor is filled in chunks of 16 blocks (1024
    tokens) along S, chunk c drawn from child stream c of its tensor's stream
    (so chunks can be filled by parallel threads and the result is still a
    fixed function of the seed);
  * m_* has shape [B, h, s1, D] with per-component N(0, sigma^2) entries; for
    the AR(1) configurations m[t] = rho*m[t-1] + sqrt(1-rho^2)*sigma*z along
    the t axis of the (T, H, W) block grid, m[0] = sigma*z;
  * q[b, s, h, :] = m_q[b, h, s // 64, :] + n_q[b, s, h, :], n ~ N(0, 1);
    k likewise; v ~ N(0, 1);
  * bf16 configurations are rounded to nearest-even bf16, the fp32 one is
    kept in fp32.
Block index inside the grid is raster order b = (t*H + y)*W + x.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Tuple

import numpy as np

BLOCK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    h: int
    D: int
    S: int
    grid: Tuple[int, int, int]  # (T, H, W) block grid, T*H*W == S // 64
    sigma: float
    rho: Optional[float]  # AR(1) coefficient along t, None = independent blocks
    thr: Tuple[float, ...]
    sta_half_widths: Tuple[int, int, int]  # (wt, wh, ww)
    dtype: str  # "f32" or "bf16"

    @property
    def s1(self) -> int:
        return self.S // BLOCK

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def elements(self) -> int:
        return self.B * self.S * self.h * self.D


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_f32", 1, 2, 64, 1024, (4, 2, 2), 0.5, None, (0.9,), (1, 1, 1), "f32"),
        Workload("small_bf16", 1, 8, 128, 8192, (8, 4, 4), 0.5, None, (0.9,), (1, 1, 1), "bf16"),
        Workload("480p_bf16", 1, 24, 128, 32768, (8, 8, 8), 0.75, 0.8, (0.8,), (1, 1, 1), "bf16"),
        Workload("720p_bf16", 1, 24, 128, 98304, (24, 8, 8), 0.75, 0.8, (0.9,), (3, 1, 1), "bf16"),
        Workload("sweep_bf16", 2, 16, 128, 65536, (16, 8, 8), 0.75, 0.8,
                 (0.5, 0.7, 0.9, 0.99, 1.0), (1, 1, 1), "bf16"),
    ]
}


def custom(name: str, B: int, h: int, D: int, S: int, grid, sigma=0.5, rho=None,
           thr=(0.9,), sta=(1, 1, 1), dtype="bf16") -> Workload:
    """A workload outside the fixed table (edge-case tests)."""
    assert S % BLOCK == 0 and grid[0] * grid[1] * grid[2] == S // BLOCK
    return Workload(name, B, h, D, S, tuple(grid), sigma, rho, tuple(thr), tuple(sta), dtype)


CHUNK_BLOCKS = 16


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _block_means(ss: np.random.SeedSequence, w: Workload) -> np.ndarray:
    rng = np.random.default_rng(ss)
    T, H, W = w.grid
    if w.rho is None:
        return w.sigma * rng.standard_normal((w.B, w.h, w.s1, w.D))
    z = rng.standard_normal((w.B, w.h, T, H, W, w.D))
    m = np.empty_like(z)
    m[:, :, 0] = w.sigma * z[:, :, 0]
    a = math.sqrt(1.0 - w.rho * w.rho) * w.sigma
    for t in range(1, T):
        m[:, :, t] = w.rho * m[:, :, t - 1] + a * z[:, :, t]
    return m.reshape(w.B, w.h, w.s1, w.D)


def _noise(ss: np.random.SeedSequence, w: Workload, means: Optional[np.ndarray]) -> np.ndarray:
    """N(0,1) tokens [B, S, h, D] float32 (+ block means), filled chunk by chunk."""
    x = np.empty((w.B, w.S, w.h, w.D), dtype=np.float32)
    nchunk = (w.s1 + CHUNK_BLOCKS - 1) // CHUNK_BLOCKS
    kids = ss.spawn(nchunk)
    mt = None if means is None else means.transpose(0, 2, 1, 3).astype(np.float32)  # [B,s1,h,D]

    def fill(c):
        b0, b1 = c * CHUNK_BLOCKS, min(w.s1, (c + 1) * CHUNK_BLOCKS)
        rng = np.random.default_rng(kids[c])
        part = rng.standard_normal((w.B, (b1 - b0) * BLOCK, w.h, w.D), dtype=np.float32)
        if mt is not None:
            pv = part.reshape(w.B, b1 - b0, BLOCK, w.h, w.D)
            pv += mt[:, b0:b1, None, :, :]
        x[:, b0 * BLOCK:b1 * BLOCK] = part

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(nchunk)))
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16, returned as uint16 bit patterns."""
    src = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(src.shape, dtype=np.uint16)
    step = 1 << 22

    def conv(i):
        b = src[i:i + step].view(np.uint32)
        r = ((b >> 16) & 1) + np.uint32(0x7FFF)
        out[i:i + step] = ((b + r) >> 16).astype(np.uint16)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(conv, range(0, src.size, step)))
    return out.reshape(np.shape(x))


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def generate(w: Workload, seed: int = 0) -> Dict[str, np.ndarray]:
    """Draw q, k, v for a workload.

    Returns a dict with "q", "k", "v" in the storage type the GPU reads:
    float32 arrays for "f32" workloads, uint16 bf16 bit patterns for "bf16".
    Shapes are [B, S, h, D], C-contiguous.
    """
    s_mq, s_nq, s_mk, s_nk, s_v = np.random.SeedSequence(seed).spawn(5)
    out = {"q": _noise(s_nq, w, _block_means(s_mq, w)),
           "k": _noise(s_nk, w, _block_means(s_mk, w)),
           "v": _noise(s_v, w, None)}
    if w.dtype == "bf16":
        out = {n: f32_to_bf16_bits(a) for n, a in out.items()}
    return out


def generate_dout(w: Workload, seed: int = 0) -> np.ndarray:
    """An upstream gradient for the backward: N(0,1) tokens [B, S, h, D] drawn
    from its own stream (SeedSequence((seed, 1))), in the workload's storage type."""
    x = _noise(np.random.SeedSequence((seed, 1)), w, None)
    return f32_to_bf16_bits(x) if w.dtype == "bf16" else x


def as_float(x: np.ndarray) -> np.ndarray:
    """Storage array (float32 or bf16 bits) -> exact float32 values."""
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x)
    return np.asarray(x, dtype=np.float32)


def random_sta(rng: np.random.Generator, s1: int, density: float) -> np.ndarray:
    """A random 0/1 block mask for edge-case tests (not a window)."""
    return (rng.random((s1, s1)) < density).astype(np.uint8)
