"""Seeded input generators.

Every value any test or benchmark feeds to the collectives comes from here, drawn with
numpy's PCG64 from an explicit seed. bf16 tensors are carried as uint16 bit patterns.

To keep this module free of the method's arithmetic, float32 draws are turned into bf16
by TRUNCATION (keep the upper 16 bits of the binary32 pattern), not by the
round-to-nearest-even that the reduce step uses on its sums. The values are still drawn
from the stated distributions (uniform[-1,1], N(0,1)) up to that truncation.
"""

from __future__ import annotations

import numpy as np


def seeded_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def bf16_bits_from_f32_trunc(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of each binary32 pattern (round toward zero)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def uniform_f32(rng: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def uniform_bf16(rng: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return bf16_bits_from_f32_trunc(uniform_f32(rng, shape, lo, hi))


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits_from_f32_trunc(normal_f32(rng, shape))


def small_int_f32(rng: np.random.Generator, shape, lim=16) -> np.ndarray:
    """Integers in [-lim, lim] as float32 (sums of a few of them are exact)."""
    return rng.integers(-lim, lim + 1, size=shape).astype(np.float32)


def small_int_bf16(rng: np.random.Generator, shape, lim=16) -> np.ndarray:
    """Integers in [-lim, lim] as bf16 bit patterns (exact: |v| <= 256 fits 8 bits)."""
    return bf16_bits_from_f32_trunc(small_int_f32(rng, shape, lim))


def random_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 256, size=shape, dtype=np.uint8)


def zipf_topk_routing(seed: int, n_ranks: int, tokens_per_rank: int, n_experts: int,
                      topk: int, s: float) -> np.ndarray:
    """Routing table [n_ranks, tokens_per_rank, topk] of expert ids (int32).

    Expert popularity follows Zipf(s): a seeded permutation gives every expert a
    popularity rank k = 1..n_experts and p(expert) is proportional to 1/k^s. Each token
    draws `topk` DISTINCT experts by sequential sampling without replacement (the chosen
    expert's mass is removed and the rest renormalised). The sampling is done with the
    Gumbel-top-k trick, which gives exactly that sequential law: the k largest of
    log p_e + Gumbel noise, in descending order.
    """
    rng = seeded_rng(seed)
    perm = rng.permutation(n_experts)
    pop_rank = np.empty(n_experts, dtype=np.float64)
    pop_rank[perm] = np.arange(1, n_experts + 1, dtype=np.float64)
    logp = -s * np.log(pop_rank)
    g = rng.gumbel(size=(n_ranks, tokens_per_rank, n_experts))
    keys = logp[None, None, :] + g
    top = np.argsort(-keys, axis=-1, kind="stable")[..., :topk]
    return top.astype(np.int32)


def random_naming(rng: np.random.Generator, n_ranks: int, max_len: int, max_segs: int,
                  n_names: int, op: str):
    """A random well-formed naming for small brute-force comparisons.

    Returns (in_len, in_segs, out_len, out_segs), segments as (rank, offset, count, name).
    Names get a random count each; producers are drawn at random input places
    (overlapping producers allowed); consumers are placed without overlap per rank.
    For op == "copy" each consumed name gets exactly one producer.
    """
    in_len = [int(rng.integers(1, max_len + 1)) for _ in range(n_ranks)]
    out_len = [int(rng.integers(1, max_len + 1)) for _ in range(n_ranks)]
    counts = {}
    in_segs = []
    for name in range(n_names):
        c = int(rng.integers(1, max(2, min(in_len) + 1)))
        counts[name] = c
        n_prod = 1 if op == "copy" else int(rng.integers(1, max_segs + 1))
        for _ in range(n_prod):
            r = int(rng.integers(0, n_ranks))
            if in_len[r] < c:
                r = int(np.argmax(in_len))
            off = int(rng.integers(0, in_len[r] - c + 1))
            in_segs.append((r, off, c, name))
    out_segs = []
    for r in range(n_ranks):
        pos = 0
        for _ in range(max_segs):
            name = int(rng.integers(0, n_names))
            c = counts[name]
            gap = int(rng.integers(0, 3))
            if pos + gap + c > out_len[r]:
                break
            out_segs.append((r, pos + gap, c, name))
            pos += gap + c
    return in_len, in_segs, out_len, out_segs


def _device_trunc_bf16(torch, x):
    """float32 device tensor -> bf16 bit patterns (int16), by the same truncation as
    ``bf16_bits_from_f32_trunc`` (the upper 16 bits of each binary32 pattern)."""
    return (x.view(torch.int32) >> 16).to(torch.int16)


def device_uniform_bf16(torch, seed: int, shape, device, lo=-1.0, hi=1.0):
    """uniform[lo, hi) bf16 patterns (int16 tensor) drawn on the device by torch's generator
    seeded with `seed`: the recipe for inputs of hundreds of MiB per rank, which numpy would
    take minutes to draw. Same distribution and truncation as ``uniform_bf16``; another
    random stream."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.rand(shape, device=device, generator=g, dtype=torch.float32) * (hi - lo) + lo
    return _device_trunc_bf16(torch, x)


def device_normal_bf16(torch, seed: int, shape, device):
    """N(0,1) bf16 patterns (int16 tensor) drawn on the device (see device_uniform_bf16)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return _device_trunc_bf16(torch, torch.randn(shape, device=device, generator=g,
                                                 dtype=torch.float32))
