"""Seeded synthetic workloads for the attention hot path.

This module holds the workload table and the seeded input generators, and
nothing else: no step of the attention method is computed here.  Both the
fp64 oracle (under ``oracle/``) and the CUDA path draw their inputs from these
functions, so the two sides see bit-identical bf16 inputs.

Shapes follow the depth -> width rule of the nanochat course guide
(ai.flicky.cc, "nanochat: свой ChatGPT от токенизатора до чата", section
"Одна ручка: --depth", step 1 and the depth table): width = 64 * depth rounded up
to a multiple of the head size 128, heads = width / 128.  d20 is also given as
"1280 hidden channels, 10 heads of 128" on 7minutos.es ("Andrej Karpathy lanza
nanochat ...", section "Modelo, escalado y objetivo de 'speedrun'").

Recipe (the pages print no attention inputs; this is the plainest synthetic
stand-in): ``torch.Generator('cpu').manual_seed(seed)``, ``torch.randn`` in
fp32, cast to bf16 with round-to-nearest-even, drawn in the order
q, k, v, dout.  Decode draws the per-stream cache lengths first
(uniform integers in [1, capacity]), then q, the raw key cache, the value
cache.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

EPS = 1e-6          # QK RMSNorm epsilon used by every workload
ROPE_BASE = 10000.0  # RoPE base used by every workload


@dataclass(frozen=True)
class AttnWorkload:
    """Causal self-attention fwd+bwd workload, tensors laid out [B, T, H, D]."""
    name: str
    B: int
    T: int
    H: int
    D: int
    seed: int
    depth: int | None = None  # nanochat --depth this shape comes from

    @property
    def width(self) -> int:
        return self.H * self.D

    def fwd_flops(self) -> float:
        """Algorithmic causal forward FLOPs: two T x T x D matmuls over half the
        score matrix (masked-out half not counted)."""
        return 4.0 * self.B * self.H * self.T * self.T * self.D / 2.0

    def fwd_bwd_flops(self) -> float:
        """Forward + backward: the backward is 2.5x the forward (five matmuls
        against the forward's two), so the total is 3.5x the forward."""
        return 3.5 * self.fwd_flops()


@dataclass(frozen=True)
class DecodeWorkload:
    """Single-token decode over a bf16 KV cache laid out [B, Tcap, H, D]."""
    name: str
    B: int
    H: int
    D: int
    Tcap: int
    seed: int


TINY = AttnWorkload("tiny", B=1, T=128, H=2, D=64, seed=0)
D12 = AttnWorkload("d12", B=8, T=2048, H=6, D=128, seed=1, depth=12)
D20 = AttnWorkload("d20", B=32, T=2048, H=10, D=128, seed=2, depth=20)
D26 = AttnWorkload("d26", B=16, T=2048, H=13, D=128, seed=3, depth=26)
D20_DECODE = DecodeWorkload("d20_decode", B=32, H=10, D=128, Tcap=2048, seed=4)

ATTN_WORKLOADS = {w.name: w for w in (TINY, D12, D20, D26)}
DECODE_WORKLOADS = {D20_DECODE.name: D20_DECODE}


def depth_to_shape(depth: int, aspect: int = 64, head_dim: int = 128) -> tuple[int, int]:
    """(width, heads) from --depth: width = depth*aspect rounded up to a
    multiple of head_dim; heads = width / head_dim."""
    width = -(-depth * aspect // head_dim) * head_dim
    return width, width // head_dim


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    """N(0,1) drawn in fp32 from ``gen`` and rounded to bf16 (RNE)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def attn_inputs(B: int, T: int, H: int, D: int, seed: int, with_dout: bool = True, kv_heads: int | None = None):
    """q, k, v (and dout) as bf16 CPU tensors [B, T, H, D], drawn in that order
    (k and v with kv_heads heads when given)."""
    g = _gen(seed)
    Hkv = H if kv_heads is None else kv_heads
    q = randn_bf16((B, T, H, D), g)
    k = randn_bf16((B, T, Hkv, D), g)
    v = randn_bf16((B, T, Hkv, D), g)
    dout = randn_bf16((B, T, H, D), g) if with_dout else None
    return q, k, v, dout


def workload_inputs(w: AttnWorkload, with_dout: bool = True):
    return attn_inputs(w.B, w.T, w.H, w.D, w.seed, with_dout)


def decode_inputs(B: int, H: int, D: int, Tcap: int, seed: int, lens=None, kv_heads: int | None = None):
    """lens [B] int32 (uniform in [1, Tcap] unless given), then q [B,H,D],
    raw keys [B,Tcap,Hkv,D] and values [B,Tcap,Hkv,D] (Hkv = kv_heads, default
    H), all bf16 CPU tensors.

    ``lens[b]`` counts the valid cache slots of stream b including the new
    token, whose position is ``lens[b] - 1``.  The raw key at that slot is the
    new token's key.
    """
    g = _gen(seed)
    if lens is None:
        lens = torch.randint(1, Tcap + 1, (B,), generator=g, dtype=torch.int64)
    lens = torch.as_tensor(lens, dtype=torch.int32)
    Hkv = H if kv_heads is None else kv_heads
    q = randn_bf16((B, H, D), g)
    k_raw = randn_bf16((B, Tcap, Hkv, D), g)
    v = randn_bf16((B, Tcap, Hkv, D), g)
    return lens, q, k_raw, v


def prefill_inputs(B: int, C: int, H: int, D: int, Tcap: int, seed: int, start=None, kv_heads: int | None = None):
    """start [B] int32 (uniform in [0, Tcap - C] unless given), then the chunk's
    queries q [B,C,H,D], raw keys [B,Tcap,Hkv,D] and values [B,Tcap,Hkv,D]
    (Hkv = kv_heads, default H), all bf16 CPU tensors.  Stream b's chunk holds positions start[b] .. start[b]+C-1;
    its own raw keys and values are the slots start[b] .. start[b]+C-1 of
    k_raw and v, the slots before them the stream's history."""
    g = _gen(seed)
    if start is None:
        start = torch.randint(0, Tcap - C + 1, (B,), generator=g, dtype=torch.int64)
    start = torch.as_tensor(start, dtype=torch.int32)
    Hkv = H if kv_heads is None else kv_heads
    q = randn_bf16((B, C, H, D), g)
    k_raw = randn_bf16((B, Tcap, Hkv, D), g)
    v = randn_bf16((B, Tcap, Hkv, D), g)
    return start, q, k_raw, v


def decode_workload_inputs(w: DecodeWorkload, kv_heads: int | None = None):
    return decode_inputs(w.B, w.H, w.D, w.Tcap, w.seed, kv_heads=kv_heads)


def decode_bytes(lens, H: int, D: int, kv_heads: int | None = None) -> int:
    """Algorithmic HBM bytes of one decode step: every valid K and V cache
    row read once (16-bit; kv_heads of them per slot, default H), plus q, out
    and lens."""
    Hkv = H if kv_heads is None else kv_heads
    n = int(torch.as_tensor(lens).to(torch.int64).sum())
    B = int(torch.as_tensor(lens).numel())
    return n * Hkv * D * 2 * 2 + 2 * B * H * D * 2 + 4 * B
