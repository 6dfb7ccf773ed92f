"""Seeded synthetic inputs for the Hybrid-SWA dual-pool workloads.

This module only draws numbers: sequence lengths, free-list orders and the
Gaussian Q/K/V values. It holds none of the attention or pool arithmetic, so
that both the CPU oracle (``oracle/``) and the CUDA library can be fed from it
without sharing any of the method's code.

The five workloads follow the serving shapes described in "MiMo-V2.5 Series
Inference Full-Link Optimization" (Sec. 1.1: 70 layers = 10 Full + 60 SWA,
window 128; Sec. 4.2: chunked prefill over long cached prefixes; Sec. 2.1:
dual pool and transfer by SWA mask).  No public dataset is involved; every
value is drawn from a fixed seed.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

KIND_FULL = 0
KIND_SWA = 1

DTYPE_F32 = 0
DTYPE_BF16 = 1

TORCH_DTYPE = {DTYPE_F32: torch.float32, DTYPE_BF16: torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    window: int
    dtype: int
    # cached lengths before the step (one entry per sequence)
    cached: tuple
    # tokens appended per sequence in one step (1 for decode, C for prefill)
    n_new: int
    layer_kinds: tuple


def _uniform_lengths(n, lo, hi, seed):
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


def lognormal_lengths(n, median, sigma, cap, seed):
    """Lengths ~ lognormal(ln median, sigma), rounded, clipped to [1, cap]."""
    rng = np.random.default_rng(seed)
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return tuple(int(v) for v in np.clip(np.rint(x), 1, cap))


def tiny():
    """2 seqs (300 and 77 cached), 4 Q / 1 KV heads, d 64, page 16, fp32."""
    return Workload("tiny", 1, 4, 1, 64, 16, 128, DTYPE_F32, (300, 77), 1,
                    (KIND_FULL, KIND_SWA))


def decode_batch(n_seqs=64):
    """64 seqs, cached lengths uniform in [1024, 32768], 64/8 heads, d 128."""
    return Workload("decode_batch", 2, 64, 8, 128, 64, 128, DTYPE_BF16,
                    _uniform_lengths(n_seqs, 1024, 32768, 2), 1,
                    (KIND_FULL, KIND_SWA))


def chunked_prefill(n_seqs=8, chunk=4096):
    """8 seqs, cached prefix uniform in [8192, 65536], 4096-token chunk."""
    return Workload("chunked_prefill", 3, 64, 8, 128, 64, 128, DTYPE_BF16,
                    _uniform_lengths(n_seqs, 8192, 65536, 3), chunk,
                    (KIND_FULL, KIND_SWA))


def hybrid70(n_seqs=128, context=131072):
    """70 layers (Full at every 7th), batch 128 at 128K cached tokens each."""
    kinds = tuple(KIND_FULL if (i % 7) == 6 else KIND_SWA for i in range(70))
    return Workload("hybrid70", 4, 64, 8, 128, 64, 128, DTYPE_BF16,
                    (context,) * n_seqs, 1, kinds)


def swa_transfer(n_seqs=256):
    """256 seqs, lognormal lengths (median 16K, sigma 1.0, cap 256K), 60 SWA layers."""
    return Workload("swa_transfer", 5, 64, 8, 128, 64, 128, DTYPE_BF16,
                    lognormal_lengths(n_seqs, 16384, 1.0, 262144, 5), 1,
                    (KIND_SWA,) * 60)


def permutation(n, seed):
    """A seeded permutation of range(n) as int32 (free-list order)."""
    rng = np.random.default_rng(seed)
    return rng.permutation(n).astype(np.int32)


def normal(shape, seed, dtype, device="cpu"):
    """N(0, 1) values drawn in fp32 from a seeded generator, then cast."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    return x.to(TORCH_DTYPE[dtype] if isinstance(dtype, int) else dtype)
