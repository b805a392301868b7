"""Seeded synthetic inputs for the attention forward pass.

This module draws random numbers and rounds them to bf16 or fp16; it holds none of
the attention arithmetic.  It is the one module that both the CUDA path's
callers (tests, benchmark) and the oracle's callers use, so that both sides
see the same bf16 bit patterns.

Recipe (the pages measure on no dataset; these tensors stand in for the
"random Q, K, V" of the self-check in "FlashAttention 怎么做?online softmax
怎么更新?", section 手撕代码, at the workload shapes below):

* every tensor is laid out [B, H, N, d] (BHSD) and drawn in the order Q, K, V;
* each tensor is cut into chunks of ``CHUNK`` elements in row-major order;
  chunk c of tensor t (0 = Q, 1 = K, 2 = V) comes from its own counter-based
  Philox stream keyed by (seed, t, c), so the bits do not depend on the
  number of threads or on the machine;
* "normal(std)" draws float32 standard normals times std, "uniform" draws
  float32 U[0, 1) mapped to [-1, 1);
* the float32 samples are rounded to bf16 (or, on request, fp16) with
  round-to-nearest-even.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

CHUNK = 1 << 22


@dataclass(frozen=True)
class Workload:
    """One attention problem: sizes, masking, scale and input distributions."""

    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    qk_dist: str = "normal"
    qk_std: float = 1.0
    v_dist: str = "normal"
    seed: int = 0

    @property
    def scale(self) -> float:
        # the pages' default, 1/sqrt(d), rounded once to float32
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def flops(self) -> float:
        # 2 GEMMs of 2*Nq*Nk*d each per (b, h); causal keeps about half
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2 if self.causal else f


# The five workloads: a one-tile case, a ragged non-tile-multiple case, two
# causal long-sequence cases and a short-query / long-key cross-length case.
WORKLOADS = [
    Workload("b1_h1_n128_d64", 1, 1, 128, 128, 64, False, seed=1),
    Workload("b2_h8_n1000_d64", 2, 8, 1000, 1000, 64, False, seed=2),
    Workload("b4_h16_n4096_d128_causal", 4, 16, 4096, 4096, 128, True, seed=3),
    Workload("b1_h32_n16384_d128_causal", 1, 32, 16384, 16384, 128, True,
             v_dist="uniform", seed=4),
    Workload("b16_h32_nq128_nk8192_d128", 16, 32, 128, 8192, 128, False,
             qk_std=2.0, seed=5),
]


# Further measured shapes beyond the five: a long causal sequence at head
# dimension 256 (the largest head size in the arithmetic-intensity table of
# "Flash Attention 全解析(上)", section 1), with the same FLOP count as the
# 16384-length d=128 case, and a long non-causal sequence at d=128.
EXTRA_WORKLOADS = [
    Workload("b1_h16_n16384_d256_causal", 1, 16, 16384, 16384, 256, True, seed=6),
    # the non-causal counterpart of the 16384-length causal case (B=1, H=32,
    # d=128, the shape of the utilisation table in "FlashAttention-2 算法架构升级",
    # section 四)
    Workload("b1_h32_n16384_d128", 1, 32, 16384, 16384, 128, False, v_dist="uniform", seed=7),
]


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    for w in WORKLOADS + EXTRA_WORKLOADS:
        if w.name == name_or_index:
            return w
    raise KeyError(name_or_index)


def _fill_chunk(out: np.ndarray, seed: int, tensor_id: int, chunk: int, dist: str, std: float):
    rng = np.random.Generator(np.random.Philox(key=[seed, (tensor_id << 32) | chunk]))
    if dist == "normal":
        rng.standard_normal(out=out, dtype=np.float32)
        if std != 1.0:
            out *= np.float32(std)
    elif dist == "uniform":
        rng.random(out=out, dtype=np.float32)
        out *= np.float32(2.0)
        out -= np.float32(1.0)
    else:
        raise ValueError(f"unknown distribution {dist!r}")


def draw_bf16(shape, seed: int, tensor_id: int, dist: str = "normal", std: float = 1.0,
              threads: int | None = None, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """One seeded tensor of the given shape, rounded (nearest even) to `dtype`,
    bf16 by default or fp16 (CPU, contiguous)."""
    n = int(np.prod(shape)) if len(shape) else 1
    buf = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK
    jobs = [(c, buf[c * CHUNK:min(n, (c + 1) * CHUNK)]) for c in range(nchunks)]
    threads = threads or min(16, os.cpu_count() or 1)
    if nchunks <= 1 or threads <= 1:
        for c, view in jobs:
            _fill_chunk(view, seed, tensor_id, c, dist, std)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda job: _fill_chunk(job[1], seed, tensor_id, job[0], dist, std), jobs))
    return torch.from_numpy(buf).to(dtype).reshape(shape)


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int, seed: int, qk_dist: str = "normal",
             qk_std: float = 1.0, v_dist: str = "normal", threads: int | None = None,
             dtype: torch.dtype = torch.bfloat16):
    """Q [B,H,Nq,d], K and V [B,H,Nk,d] as bf16 (or fp16) CPU tensors drawn from ``seed``."""
    Q = draw_bf16((B, H, Nq, d), seed, 0, qk_dist, qk_std, threads, dtype)
    K = draw_bf16((B, H, Nk, d), seed, 1, qk_dist, qk_std, threads, dtype)
    V = draw_bf16((B, H, Nk, d), seed, 2, v_dist, 1.0, threads, dtype)
    return Q, K, V


def workload_inputs(w: Workload, threads: int | None = None):
    return make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed, w.qk_dist, w.qk_std, w.v_dist, threads)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bit patterns of a CPU bf16 (or fp16) tensor, as a uint16 array (no copy)."""
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("expected a bf16 or fp16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
