"""Seeded synthetic inputs shaped like the MiniMax-01 lightning-attention
workload (64 heads of dimension 128, long contexts).

This module holds input recipes only -- no arithmetic of the method -- so both
the CUDA path and the CPU oracle can be fed the same tensors.

Recipe (all draws from a ``torch.Generator`` seeded explicitly):
  * q, k, v ~ N(0, 1) in fp32; q and k are then multiplied by d^-1/2; the
    result is cast to the compute dtype (bf16, or kept fp32).
  * per-head decay lambda_h = exp(-2^(-8 (h + 1) / H)); for H = 64 this runs
    from about 0.3997 (head 0) to about 0.9961 (head 63); for H = 1 it is
    exp(-2^-8).
  * varlen: sequence lengths uniform in [lo, hi] (``torch.randint``), packed
    back to back, ``cu_seqlens`` = int32 exclusive prefix sum.
  * decode: state ~ N(0, 1) * 0.02 in fp32, one fresh token per sequence.
  * cached states a prefill continues from: ~ N(0, 1) * 0.3 in fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


def decay_schedule(num_heads: int) -> torch.Tensor:
    """lambda_h = exp(-2^(-8 (h+1) / H)) as fp32 [H]."""
    h = torch.arange(num_heads, dtype=torch.float64)
    lam = torch.exp(-torch.pow(2.0, -8.0 * (h + 1.0) / num_heads))
    return lam.to(torch.float32)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _qkv(g, shape, dtype, device):
    d = shape[-1]
    scale = 1.0 / math.sqrt(d)
    q = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * scale
    k = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * scale
    v = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    return q.to(dtype), k.to(dtype), v.to(dtype)


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H, d]
    k: torch.Tensor
    v: torch.Tensor
    decay: torch.Tensor        # [H] fp32
    cu_seqlens: torch.Tensor   # [nseq + 1] int32

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.numel() - 1)


def cu_from_lengths(lengths) -> torch.Tensor:
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def varlen_lengths(num_seqs: int = 16, lo: int = 1024, hi: int = 32768,
                   seed: int = 0) -> torch.Tensor:
    """Sequence lengths uniform in [lo, hi] (int64, CPU)."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (num_seqs,), generator=g)


def prefill_inputs(lengths, num_heads: int, head_dim: int,
                   dtype=torch.bfloat16, seed: int = 0, device="cpu",
                   decay: torch.Tensor | None = None) -> PrefillInputs:
    """Packed q, k, v for sequences of the given lengths."""
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    g = _gen(seed, device)
    q, k, v = _qkv(g, (T, num_heads, head_dim), dtype, device)
    lam = decay_schedule(num_heads) if decay is None else decay.to(torch.float32)
    return PrefillInputs(q, k, v, lam.to(device), cu.to(device))


def cached_states(num_seqs: int, num_heads: int, head_dim: int, std: float = 0.3,
                  seed: int = 0, device="cpu") -> torch.Tensor:
    """A seeded stand-in for a prefix KV cache: fp32 [nseq, H, d, d] ~ N(0, std^2)."""
    g = _gen(seed, device)
    return torch.randn((num_seqs, num_heads, head_dim, head_dim), generator=g,
                       dtype=torch.float32, device=device) * std


@dataclass
class DecodeInputs:
    q: torch.Tensor        # [steps, B, H, d] (or [B, H, d] for one step)
    k: torch.Tensor
    v: torch.Tensor
    decay: torch.Tensor    # [H]
    state: torch.Tensor    # [B, H, d, d] fp32


def decode_inputs(batch: int, num_heads: int, head_dim: int, steps: int = 1,
                  dtype=torch.bfloat16, seed: int = 0, device="cpu",
                  state_std: float = 0.02) -> DecodeInputs:
    g = _gen(seed, device)
    st = torch.randn((batch, num_heads, head_dim, head_dim), generator=g,
                     dtype=torch.float32, device=device) * state_std
    q, k, v = _qkv(g, (steps, batch, num_heads, head_dim), dtype, device)
    return DecodeInputs(q, k, v, decay_schedule(num_heads).to(device), st)


# The workloads this library is measured and checked on.
TINY = dict(name="tiny", lengths=[256], num_heads=1, head_dim=64,
            dtype=torch.float32, chunk=64)
PREFILL_8K = dict(name="prefill_8k", lengths=[8192], num_heads=64,
                  head_dim=128, dtype=torch.bfloat16)
PREFILL_128K = dict(name="prefill_128k", lengths=[131072], num_heads=64,
                    head_dim=128, dtype=torch.bfloat16)
VARLEN_16 = dict(name="varlen_16", num_seqs=16, lo=1024, hi=32768,
                 num_heads=64, head_dim=128, dtype=torch.bfloat16)
DECODE_128 = dict(name="decode_128", batch=128, num_heads=64, head_dim=128,
                  steps=1000, dtype=torch.bfloat16)
