"""Seeded synthetic inputs for the per-token decoder path.

This module only draws numbers: it holds none of the operators' arithmetic.
The same bytes feed the CUDA library and the CPU oracle. Every tensor is made
on the host from ``numpy.random.default_rng(SeedSequence([seed, stream]))``,
drawn in fp32 and quantised to the target dtype with torch's
round-to-nearest-even conversion.

Distributions follow the workloads the pages measure on:
activations ~N(0, 1), RMSNorm weights ~N(1, 0.1), residuals ~N(0, 0.5),
positions uniform in [0, max_pos), slot_mapping = the first T entries of a
seeded permutation of the cache's slots, KV cache prefilled with a sentinel.

The RoPE cos/sin tables are inputs to the operator: ``rope_tables`` builds the
usual neox frequency tables cos(p * theta^(-2i/head_dim)) in float64 and rounds
them to fp32, as a caller's model would precompute them (m.lsln.cn "21 个算子"
section 2.3 recommends precomputed caches).
"""
from __future__ import annotations

import numpy as np
import torch

SENTINEL_BF16 = 0xDEAD  # bit pattern prefilled into every KV-cache element


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


def normal(shape, mean: float, std: float, dtype: torch.dtype, seed: int, stream: int) -> torch.Tensor:
    """A CPU tensor of ``dtype`` with N(mean, std) entries (drawn in fp32, then rounded)."""
    g = rng(seed, stream)
    a = g.standard_normal(size=tuple(shape), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return torch.from_numpy(a).to(dtype)


def positions(T: int, max_pos: int, seed: int, stream: int) -> torch.Tensor:
    return torch.from_numpy(rng(seed, stream).integers(0, max_pos, size=T, dtype=np.int64))


def slots(T: int, capacity: int, seed: int, stream: int) -> torch.Tensor:
    """T distinct slots: a prefix of a seeded permutation of range(capacity)."""
    if T > capacity:
        raise ValueError("more tokens than cache slots")
    return torch.from_numpy(rng(seed, stream).permutation(capacity)[:T].astype(np.int64))


def rope_tables(max_pos: int, head_dim: int, theta: float) -> tuple[torch.Tensor, torch.Tensor]:
    """fp32 cos/sin tables of shape [max_pos, head_dim // 2]."""
    half = head_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return (torch.from_numpy(np.cos(ang).astype(np.float32)),
            torch.from_numpy(np.sin(ang).astype(np.float32)))


def sentinel_cache(shape, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """A cache tensor whose every element holds the sentinel bit pattern."""
    if dtype == torch.float32:
        bits = torch.full(tuple(shape), 0x7FBADBAD, dtype=torch.int32)
        return bits.view(torch.float32)
    bits = torch.full(tuple(shape), SENTINEL_BF16 - 0x10000, dtype=torch.int16)
    return bits.view(dtype)


# ---------------------------------------------------------------------------
# Workloads (sizes of the pages' models; seed = 1000 + workload index)
# ---------------------------------------------------------------------------

QWEN25_15B = dict(hidden=1536, n_head=12, n_kv_head=2, head_dim=128, intermediate=8960,
                  layers=28, rope_theta=1e6, max_pos=32768)
LLAMA3_8B_MLP = dict(intermediate=14336)
RMS_SWEEP_D = (128, 512, 1024, 1536, 2048, 2176, 4096, 8192)
RMS_SWEEP_ROWS = 512
ADD_RMS_T = (1, 16, 256, 4096)
ROPE_T = (1, 64, 2048)
GLU_T = (1, 64, 512, 4096)
CACHE_BLOCKS, CACHE_BLOCK_SIZE = 4096, 16
EPS = 1e-6


def rms_inputs(rows: int, D: int, dtype: torch.dtype, seed: int):
    x = normal((rows, D), 0.0, 1.0, dtype, seed, 1)
    w = normal((D,), 1.0, 0.1, dtype, seed, 2)
    return x, w


def add_rms_inputs(T: int, D: int, dtype: torch.dtype, seed: int):
    x = normal((T, D), 0.0, 1.0, dtype, seed, 1)
    res = normal((T, D), 0.0, 0.5, dtype, seed, 3)
    w = normal((D,), 1.0, 0.1, dtype, seed, 2)
    return x, res, w


def rope_inputs(T: int, seed: int, n_head: int = 12, n_kv_head: int = 2, head_dim: int = 128,
                num_blocks: int = CACHE_BLOCKS, block_size: int = CACHE_BLOCK_SIZE,
                max_pos: int = 32768, theta: float = 1e6, dtype: torch.dtype = torch.bfloat16,
                tables=None):
    q = normal((T, n_head, head_dim), 0.0, 1.0, dtype, seed, 11)
    k = normal((T, n_kv_head, head_dim), 0.0, 1.0, dtype, seed, 12)
    v = normal((T, n_kv_head, head_dim), 0.0, 1.0, dtype, seed, 13)
    cos, sin = tables if tables is not None else rope_tables(max_pos, head_dim, theta)
    pos = positions(T, max_pos, seed, 14)
    slot = slots(T, num_blocks * block_size, seed, 15)
    cache = sentinel_cache((2, num_blocks, block_size, n_kv_head, head_dim), dtype)
    return dict(q=q, k=k, v=v, cos=cos, sin=sin, pos=pos, slot_mapping=slot, kv_cache=cache)


def glu_inputs(T: int, I: int, dtype: torch.dtype, seed: int):
    return normal((T, 2 * I), 0.0, 1.0, dtype, seed, 21)


def uniform(shape, lo: float, hi: float, seed: int, stream: int) -> torch.Tensor:
    """An fp32 CPU tensor with U(lo, hi) entries."""
    a = rng(seed, stream).uniform(lo, hi, size=tuple(shape)).astype(np.float32)
    return torch.from_numpy(a)


def uclip_params(D: int, alpha_per_channel: bool, gamma_per_channel: bool, seed: int):
    """fp32 alpha ~ U(0.25, 1) and gamma ~ N(1, 0.1), D entries each or one.

    With x ~ N(0, 1) a fraction of alpha * x lies outside [-1, 1], so both the
    clipped and the linear part of the clamp are exercised."""
    alpha = uniform((D if alpha_per_channel else 1,), 0.25, 1.0, seed, 31)
    gamma = normal((D if gamma_per_channel else 1,), 1.0, 0.1, torch.float32, seed, 32)
    return alpha, gamma


def qkv_inputs(T: int, n_head: int, n_kv_head: int, head_dim: int, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """A fused QKV projection output [T, n_head + 2 * n_kv_head, head_dim] ~ N(0, 1)."""
    return normal((T, n_head + 2 * n_kv_head, head_dim), 0.0, 1.0, dtype, seed, 33)


def attention_inputs(B: int, lens, n_head: int, n_kv_head: int, head_dim: int, block_size: int,
                     num_blocks: int, dtype: torch.dtype, seed: int, max_blocks: int | None = None):
    """A decode batch over a paged cache: q [B, n_head, head_dim] ~ N(0, 1), a cache
    [2, num_blocks, block_size, n_kv_head, head_dim] ~ N(0, 1) (K and V), int32 seq_lens
    (`lens`: one length for every request or a sequence of B lengths), and an int32
    block table that gives each request its own blocks, drawn from a seeded permutation
    of the cache's blocks (unused table entries hold further blocks of the permutation)."""
    lens = [int(lens)] * B if np.isscalar(lens) else [int(x) for x in lens]
    need = max([(L + block_size - 1) // block_size for L in lens] + [1])
    if max_blocks is None:
        max_blocks = need
    if B * max_blocks > num_blocks:
        raise ValueError("cache too small for the requests' blocks")
    q = normal((B, n_head, head_dim), 0.0, 1.0, dtype, seed, 41)
    cache = normal((2, num_blocks, block_size, n_kv_head, head_dim), 0.0, 1.0, dtype, seed, 42)
    perm = rng(seed, 43).permutation(num_blocks)[:B * max_blocks].reshape(B, max_blocks)
    table = torch.from_numpy(perm.astype(np.int32))
    seq = torch.tensor(lens, dtype=torch.int32)
    return q, cache, table, seq


ATTN_B = (1, 32, 64)        # decode batch sizes
ATTN_CTX = 1024             # context length of the decode-attention micro-benchmark


def linear_weight(N: int, K: int, dtype: torch.dtype, seed: int, stream: int = 51) -> torch.Tensor:
    """A projection weight [N, K] (nn.Linear's layout) ~ N(0, 0.02), the usual initialisation scale."""
    return normal((N, K), 0.0, 0.02, dtype, seed, stream)


QWEN25_QKV = dict(K=1536, N=2048)     # ln1 -> qkv_proj: hidden 1536 -> (12 + 2 + 2) * 128
QWEN25_DOWN = dict(I=8960, N=1536)    # silu(gate) * up -> down_proj
LINEAR_B = (1, 16, 64)                # decode batch sizes
