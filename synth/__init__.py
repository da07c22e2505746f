"""Seeded synthetic inputs shaped like the MiMo-V2-Flash attention workloads.

This module only draws random numbers and integer layouts; it holds none of
the attention arithmetic.  Both the CUDA path and the oracle consume what it
makes.  All draws use ``torch.Generator`` (Philox on CUDA, MT19937 on CPU), so
a (seed, device) pair fixes every value; CPU and CUDA streams differ, so a
parity test generates on one device and copies.

Recipe (the pages publish no dataset for this path; these stand in for the
long-context prefill and the 16K-in / 1K-out MTP decode workloads):
- Q, K, V ~ N(0, 1) drawn in fp32 then rounded to the I/O dtype (bf16 or fp32);
- per-head sink logits ~ N(0, 1) in fp32;
- verify context lengths ~ Uniform[lo, hi] integers;
- the GA page table is a seeded random permutation of the page pool.
"""
from __future__ import annotations

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(int(seed))


def normal(shape, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def e4m3_codes(shape, seed: int, per_unit: float = 50.0, device="cpu") -> torch.Tensor:
    """uint8 E4M3 codes of N(0,1) * per_unit draws (torch's float8_e4m3fn cast,
    a library routine; draws clamped to the finite range first): an 8-bit
    cache whose entries, times a scale of about 1/per_unit, are ~ N(0,1)."""
    x = normal(shape, seed, torch.float32, device) * per_unit
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def kv_scales(Hkv: int, seed: int, device="cpu") -> torch.Tensor:
    """Per-kv-head fp32 cache scales, uniform in [0.01, 0.03]."""
    g = _gen(seed, device)
    return 0.01 + 0.02 * torch.rand(Hkv, generator=g, device=device)


def prefill_inputs(B: int, T: int, Hq: int, Hkv: int, D: int, seed: int,
                   dtype=torch.bfloat16, device="cpu"):
    """q [B,T,Hq,D], k/v [B,T,Hkv,D] in `dtype`; sink [Hq] fp32."""
    g = _gen(seed, device)
    q = torch.randn(B, T, Hq, D, generator=g, device=device).to(dtype)
    k = torch.randn(B, T, Hkv, D, generator=g, device=device).to(dtype)
    v = torch.randn(B, T, Hkv, D, generator=g, device=device).to(dtype)
    sink = torch.randn(Hq, generator=g, device=device)
    return q, k, v, sink


def packed_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n sequence lengths, log-uniform in [lo, hi] (a serving batch of prompts
    of mixed length), int32."""
    rng = np.random.Generator(np.random.Philox(int(seed)))
    x = np.exp(rng.uniform(np.log(lo), np.log(hi + 1), size=n))
    return np.clip(np.floor(x), lo, hi).astype(np.int32)


def packed_inputs(lens, Hq: int, Hkv: int, D: int, seed: int, dtype=torch.bfloat16,
                  device="cpu"):
    """A packed batch: q [total,Hq,D], k/v [total,Hkv,D] in `dtype`, sink [Hq]
    fp32 and cu_seqlens [B+1] int32 (numpy) with cu[0] = 0."""
    lens = np.asarray(lens, np.int64)
    total = int(lens.sum())
    g = _gen(seed, device)
    q = torch.randn(total, Hq, D, generator=g, device=device).to(dtype)
    k = torch.randn(total, Hkv, D, generator=g, device=device).to(dtype)
    v = torch.randn(total, Hkv, D, generator=g, device=device).to(dtype)
    sink = torch.randn(Hq, generator=g, device=device)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, sink, cu


def sink_logits(Hq: int, seed: int, device="cpu") -> torch.Tensor:
    return torch.randn(Hq, generator=_gen(seed, device), device=device)


def context_lengths(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """B integers ~ Uniform[lo, hi] (inclusive), int32."""
    rng = np.random.Generator(np.random.Philox(int(seed)))
    return rng.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)


def accept_counts(n: int, q_len: int, seed: int) -> np.ndarray:
    """n accepted-draft counts in [0, q_len-1] for a synthetic MTP walk."""
    rng = np.random.Generator(np.random.Philox(int(seed)))
    return rng.integers(0, q_len, size=n, dtype=np.int64).astype(np.int32)


def page_permutation(num_pages: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.Philox(int(seed)))
    return rng.permutation(num_pages).astype(np.int32)


def history(L: int, Hkv: int, D: int, seed: int, dtype=torch.bfloat16, device="cpu"):
    """One request's keys and values by position, [L,Hkv,D] each, drawn from
    its own seed so that any request can be regenerated alone."""
    g = _gen(seed, device)
    k = torch.randn(L, Hkv, D, generator=g, device=device).to(dtype)
    v = torch.randn(L, Hkv, D, generator=g, device=device).to(dtype)
    return k, v


def cu_seqlens(q_lens) -> np.ndarray:
    q_lens = np.asarray(q_lens, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)


def hybrid_layer_kinds(blocks: int = 8, swa_per_block: int = 5) -> list[str]:
    """Attention kind of each layer of the hybrid stack, in model order: M = 8
    blocks of 5 SWA layers followed by one GA layer, where the first layer of
    the stack is GA instead of SWA (technical-report summary, section
    "MiMo-V2-Flash Model Architecture", and its hyper-parameter paragraph:
    48 layers, 39 SWA and 9 GA).  A workload shape, not arithmetic."""
    kinds = (["swa"] * swa_per_block + ["ga"]) * blocks
    kinds[0] = "ga"
    return kinds
