"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws Q, K, V and picks
sample rows.  Both the CUDA path and the float64 oracle consume exactly the
bytes it returns.

Recipe: Q, K, V are i.i.d. N(0, 1) float32 drawn on the CPU from a seeded
``torch.Generator`` (Q for all heads, then K, then V, one head at a time) and
rounded to bfloat16 with round-to-nearest-even.  The long-context workload
additionally multiplies 1% of the key rows (floor(N/100) token positions, the
same for every head, chosen by ``randperm`` of a second generator seeded
``seed + 1``) by 8 after rounding; the multiplication is exact in bf16.  The
backward's upstream gradient dO is drawn the same way from a generator
seeded ``seed + 7``.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    P: int
    causal: bool
    layout: str  # "contiguous" | "striped" | "zigzag"
    seed: int
    key_boost_frac: float = 0.0  # fraction of key rows scaled by key_boost
    key_boost: float = 8.0
    Hkv: int = 0  # K/V heads for grouped-query attention (0: H)
    window: int = 0  # causal sliding window (0: none)
    doc_len: tuple = ()  # sequence packing: (min, max) document length (empty: one document)

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H

    @property
    def n(self) -> int:
        return self.N // self.P

    @property
    def layout_id(self) -> int:
        return {"contiguous": 0, "striped": 1, "zigzag": 2}[self.layout]

    def segments(self):
        """Document boundaries of the packed sequence, or None."""
        return document_bounds(self.N, self.seed, *self.doc_len) if self.doc_len else None

    def allowed_pairs_per_head(self) -> int:
        if self.doc_len:
            b = self.segments()
            lens = [y - x for x, y in zip(b[:-1], b[1:])]
            if not self.causal:
                return sum(L * L for L in lens)
            W = self.window or self.N
            return sum(min(W, L) * (min(W, L) + 1) // 2 + (L - min(W, L)) * W for L in lens)
        if self.causal and self.window > 0:
            W, N = min(self.window, self.N), self.N
            return W * (W + 1) // 2 + (N - W) * W  # row t sees min(t + 1, W) keys
        return self.N * (self.N + 1) // 2 if self.causal else self.N * self.N

    def flops(self) -> int:
        """Causal-adjusted FLOPs: 4*d per allowed (q, k) pair (QK^T and PV)."""
        return 4 * self.B * self.H * self.d * self.allowed_pairs_per_head()


WORKLOADS = {
    w.name: w
    for w in (
        Workload("noncausal-512", 1, 2, 512, 64, 4, False, "contiguous", 1000),
        Workload("contiguous-8k", 1, 8, 8192, 128, 8, True, "contiguous", 1001),
        Workload("striped-8k", 1, 8, 8192, 128, 8, True, "striped", 1001),
        Workload("zigzag-8k", 1, 8, 8192, 128, 8, True, "zigzag", 1001),
        Workload("striped-128k", 1, 16, 131072, 128, 16, True, "striped", 1003, key_boost_frac=0.01),
        Workload("striped-1m", 1, 8, 1048576, 128, 64, True, "striped", 1004),
        # the 128K workload in the zigzag layout (2P chunks of 4096 tokens)
        Workload("zigzag-128k", 1, 16, 131072, 128, 16, True, "zigzag", 1003, key_boost_frac=0.01),
        # causal sliding window of 4096 tokens over the 128K striped sequence
        Workload("swa-128k", 1, 16, 131072, 128, 16, True, "striped", 1003, key_boost_frac=0.01, window=4096),
        # sequence packing: documents of 1K-16K tokens packed into the 128K striped sequence
        Workload("packed-128k", 1, 16, 131072, 128, 16, True, "striped", 1003, key_boost_frac=0.01,
                 doc_len=(1024, 16384)),
        # grouped-query attention: 16 query heads sharing 4 K/V heads
        Workload("gqa-128k", 1, 16, 131072, 128, 16, True, "striped", 1003, key_boost_frac=0.01, Hkv=4),
        # profiling size: the 128K striped workload with 4 heads (inputs 3 x 134 MB)
        Workload("striped-128k-h4", 1, 4, 131072, 128, 16, True, "striped", 1003, key_boost_frac=0.01),
    )
}

ROW_SAMPLE_SEED = 2004


def make_qkv(B: int, H: int, N: int, d: int, seed: int, key_boost_frac: float = 0.0,
             key_boost: float = 8.0, device="cpu", pin: bool = False, Hkv: int = 0):
    """Return (q, k, v) bf16 tensors drawn as the module docstring says: q
    [B, H, N, d], k and v [B, Hkv, N, d] (Hkv = H unless given)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = []
    for x in range(3):
        heads = H if x == 0 else (Hkv or H)
        t = torch.empty((B, heads, N, d), dtype=torch.bfloat16, pin_memory=pin)
        for b in range(B):
            for h in range(heads):
                t[b, h].copy_(torch.randn((N, d), generator=g, dtype=torch.float32))
        out.append(t)
    q, k, v = out
    if key_boost_frac > 0.0:
        rows = boosted_key_rows(N, seed, key_boost_frac)
        k[:, :, rows, :] *= key_boost
    if device != "cpu":
        q, k, v = (x.to(device) for x in (q, k, v))
    return q, k, v


def make_dout(B: int, H: int, N: int, d: int, seed: int, device="cpu", pin: bool = False):
    """The upstream gradient dO for the backward: [B, H, N, d] i.i.d. N(0, 1)
    float32 from a CPU generator seeded ``seed + 7`` (one head at a time),
    rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7)
    t = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=pin)
    for b in range(B):
        for h in range(H):
            t[b, h].copy_(torch.randn((N, d), generator=g, dtype=torch.float32))
    return t.to(device) if device != "cpu" else t


def document_bounds(N: int, seed: int, min_len: int, max_len: int) -> list:
    """Sequence packing: documents of lengths drawn uniformly from
    [min_len, max_len] by a CPU generator seeded ``seed + 11``, packed until
    they cover N tokens (the last one cut at N).  Returns the boundaries
    [0, b1, .., N]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 11)
    bounds = [0]
    while bounds[-1] < N:
        length = int(torch.randint(min_len, max_len + 1, (1,), generator=g))
        bounds.append(min(N, bounds[-1] + length))
    return bounds


def boosted_key_rows(N: int, seed: int, frac: float) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    count = int(N * frac)
    return torch.randperm(N, generator=g)[:count].sort().values


def make_workload(w: Workload, device="cpu", pin: bool = False):
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.key_boost_frac, w.key_boost, device=device, pin=pin, Hkv=w.Hkv)


def expand_kv(t: torch.Tensor, H: int) -> torch.Tensor:
    """K or V with Hkv heads, repeated so that query head h sees K/V head
    h / (H / Hkv): the grouped-query sharing written out as plain multi-head
    attention (for the oracle)."""
    return t if t.shape[1] == H else t.repeat_interleave(H // t.shape[1], dim=1)


def sample_rows(N: int, count: int, seed: int = ROW_SAMPLE_SEED, extra=()) -> torch.Tensor:
    """Seeded distinct query positions (sorted), plus any ``extra`` positions."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    count = min(count, N)
    rows = torch.randperm(N, generator=g)[:count]
    if extra:
        rows = torch.cat([rows, torch.tensor([e for e in extra if 0 <= e < N], dtype=torch.long)])
    return torch.unique(rows)
