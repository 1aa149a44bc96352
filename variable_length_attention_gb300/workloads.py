"""Seeded synthetic workloads for jagged attention.

This module only draws inputs: sequence lengths, the packed offsets array and
bf16 tensors.  It holds none of the attention arithmetic, so both the fp64
oracle (tests) and the CUDA path can take their inputs from it.

The shapes and length mixes stand in for the production workloads the pages
describe (Meta ads user-history sequences; the block-attention ranking stack
with batch 1152, sequences up to about 4000 tokens, head_dim 64 or 128), which
are not available here.

Packed layout ("Optimizing Jagged Flash Attention with TLX", commentary on why
unequal lengths change the problem; n1n.ai page, jagged tensor layout): valid
tokens of all sequences are stored back to back, row-major [tokens, heads, dim],
and offsets[b] .. offsets[b+1] delimit sequence b, offsets[0] = 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


def offsets_from_lengths(lengths) -> np.ndarray:
    """Exclusive prefix sum with a leading 0 (length B+1, int32)."""
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    if out[-1] > np.iinfo(np.int32).max:
        raise ValueError("total token count does not fit int32 offsets")
    return out.astype(np.int32)


def lengths_log_uniform(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """L = round(exp(U(ln lo, ln hi))), clipped to [lo, hi]."""
    x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def lengths_log_normal(rng: np.random.Generator, n: int, median: float, sigma: float,
                       lo: int, hi: int) -> np.ndarray:
    """L = round(median * exp(sigma * N(0,1))), clipped to [lo, hi]."""
    x = median * np.exp(sigma * rng.standard_normal(n))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


@dataclass
class Workload:
    """One attention problem: its sizes and the seeds its tensors come from."""
    name: str
    mode: str                 # "jagged" (self), "broadcast" or "block"
    lengths: np.ndarray       # K/V sequence lengths
    num_heads: int
    num_kv_heads: int
    head_dim: int
    causal: bool = False
    nq: int = 0               # broadcast-Q: rows of the shared Q
    seed_base: int = 0
    bwd: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def offsets(self) -> np.ndarray:
        return offsets_from_lengths(self.lengths)

    @property
    def batch(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(np.sum(self.lengths))

    @property
    def max_len(self) -> int:
        return int(np.max(self.lengths)) if len(self.lengths) else 0

    @property
    def q_rows(self) -> int:
        return self.nq if self.mode == "broadcast" else self.total_tokens

    @property
    def o_rows(self) -> int:
        return self.batch * self.nq if self.mode == "broadcast" else self.total_tokens

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def tensors(self, device="cpu"):
        """q, k, v, dO as bf16, each drawn from N(0,1) in fp32 with its own seed.

        Seeds are seed_base + 2, 3, 4, 5 for q, k, v, dO.  torch's CPU and CUDA
        generators differ, so the same seed gives different values per device.
        """
        H, Hkv, D = self.num_heads, self.num_kv_heads, self.head_dim
        shapes = [(self.q_rows, H, D), (self.total_tokens, Hkv, D), (self.total_tokens, Hkv, D),
                  (self.o_rows, H, D)]
        out = []
        for i, shp in enumerate(shapes):
            g = torch.Generator(device=device)
            g.manual_seed(self.seed_base + 2 + i)
            out.append(torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16))
        return tuple(out)


def _rng(cfg: int) -> np.random.Generator:
    return np.random.default_rng(1000 * cfg + 1)


def tiny() -> Workload:
    """B=4 sequences of lengths 17, 64, 129, 256; H=2, head_dim 64, non-causal."""
    return Workload("tiny_jagged_B4_H2_D64", "jagged", np.array([17, 64, 129, 256]), 2, 2, 64,
                    seed_base=1000)


def jagged(causal: bool = False) -> Workload:
    """B=32 sequences, lengths log-uniform in [32, 4096], H=8, head_dim 128."""
    lens = lengths_log_uniform(_rng(2), 32, 32, 4096)
    return Workload(f"jagged_B32_loguniform32-4096_H8_D128{'_causal' if causal else ''}", "jagged",
                    lens, 8, 8, 128, causal=causal, seed_base=2000)


def broadcast() -> Workload:
    """Shared Q of 256 rows, H=4, head_dim 128, against B=256 K/V sequences with
    log-normal lengths (median 800, sigma 1.0 in log space), clipped to [16, 4000]."""
    lens = lengths_log_normal(_rng(3), 256, 800.0, 1.0, 16, 4000)
    return Workload("broadcastQ_Nq256_B256_lognormal800_H4_D128", "broadcast", lens, 4, 4, 128,
                    nq=256, seed_base=3000)


def block(head_dim: int = 128, batch: int = 1152, seq_len: int = 4032) -> Workload:
    """Block-diagonal attention: batch x seq_len tokens, 64-token blocks, H=4."""
    return Workload(f"block64_B{batch}_S{seq_len}_H4_D{head_dim}", "block",
                    np.full(batch, seq_len, dtype=np.int64), 4, 4, head_dim, seed_base=4000)


def dense(gqa: bool = False) -> Workload:
    """B=8 sequences of 8192 tokens in jagged layout, H=16, head_dim 128;
    the GQA variant has 4 K/V heads and is timed forward-only, the configuration
    it stands for being a forward one."""
    return Workload(f"dense_B8_L8192_H16{'_KV4' if gqa else ''}_D128", "jagged",
                    np.full(8, 8192, dtype=np.int64), 16, 4 if gqa else 16, 128,
                    seed_base=5000, bwd=not gqa)


def custom(lengths, num_heads, head_dim, *, num_kv_heads=None, causal=False, nq=0, mode=None,
           seed_base=9000) -> Workload:
    """Any shape, e.g. the edge cases of the tests."""
    if mode is None:
        mode = "broadcast" if nq > 0 else "jagged"
    return Workload(f"custom_{mode}", mode, np.asarray(lengths, dtype=np.int64), num_heads,
                    num_kv_heads or num_heads, head_dim, causal=causal, nq=nq, seed_base=seed_base)


def valid_pairs(w: Workload) -> int:
    """Query-key pairs that attention actually scores, summed over heads."""
    L = w.lengths.astype(np.int64)
    if w.mode == "broadcast":
        pairs = int(np.sum(L)) * w.nq
    elif w.mode == "block":
        full, tail = L // 64, L % 64
        pairs = int(np.sum(full * 64 * 64 + tail * tail))
    elif w.causal:
        pairs = int(np.sum(L * (L + 1) // 2))
    else:
        pairs = int(np.sum(L * L))
    return pairs * w.num_heads


def flops(w: Workload) -> tuple[int, int]:
    """(forward, backward) FLOPs on valid tokens: 4*D per scored pair forward
    (QK^T and PV, two FLOPs per multiply-add), 2.5x that backward (five GEMMs)."""
    f = 4 * w.head_dim * valid_pairs(w)
    return f, int(2.5 * f)
