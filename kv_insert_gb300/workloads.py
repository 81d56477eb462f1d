"""Seeded synthetic inputs of the QKV front, shared by the tests, the smoke
check and the benchmark.

This module draws random numbers and lays them out; it holds none of the
front's arithmetic (no projection, norm, RoPE or insert).  The rotary table is
an input of the op: it is built here the way a rotary-embedding module builds
its table at load time (interleaved layout, cos in columns 0..31 and sin in
32..63, base 10000), so that it looks like the tables the op reads in service.

Workload shapes follow the pages' contract: hidden size 8192, head_dim 64,
8 q heads per KV head, a BF16 cache [pages, num_kv_heads, 16, 128] (page
"vllm.models.muse_spark.nvidia.specialized_decode.runtime.cute_ops", attn2
paragraph and split_qkv), 1 <= M <= 16 tokens (page "...cutedsl.attention.
qkv_front", module docstring).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HIDDEN = 8192
HEAD_DIM = 64
Q_PER_KV = 8
PAGE_SLOTS = 16
SLOT_WIDTH = 128
ROPE_BASE = 10000.0


def columns_for(num_kv_heads: int) -> int:
    """N of the packed [q | k | v | gate] rows: (8 + 1 + 1 + 8) heads of 64 per KV head."""
    return 2 * (Q_PER_KV + 1) * num_kv_heads * HEAD_DIM


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    num_kv_heads: int
    max_pos: int
    num_pages: int
    seed: int
    x_std: float = 1.0
    outlier_rows: bool = False     # each row x100 with p = 0.01; >= 1 forced when M >= 4
    consecutive: bool = False      # positions p0..p0+M-1, slots across a page boundary

    @property
    def N(self) -> int:
        return columns_for(self.num_kv_heads)

    @property
    def heads(self) -> int:
        return self.N // HEAD_DIM

    def roofline_bytes(self) -> int:
        """Algorithmic HBM bytes of one call: W + x read, out + K/V written."""
        return (self.N * HIDDEN * 2 + self.M * HIDDEN * 2 + self.M * self.N * 2
                + self.M * self.num_kv_heads * SLOT_WIDTH * 2)

    def describe(self) -> dict:
        return {"workload": self.name, "M": self.M, "N": self.N, "hidden": HIDDEN,
                "num_kv_heads": self.num_kv_heads, "head_dim": HEAD_DIM,
                "cos_sin_rows": self.max_pos, "cache_pages": self.num_pages}


SWEEP_M = (1, 2, 3, 4, 5, 7, 8, 12, 13, 16)

WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


# single token, one KV head: N = 512 q + 64 k + 64 v + 512 gate = 1152
_add(Workload("m1_nkv1_n1152", M=1, num_kv_heads=1, max_pos=4096, num_pages=4, seed=1001))
# eight tokens, eight KV heads: N = 9216 (the headline decode shape)
_add(Workload("m8_nkv8_n9216", M=8, num_kv_heads=8, max_pos=32768, num_pages=4096, seed=1002))
# sixteen consecutive tokens of one request, slots crossing a page boundary
_add(Workload("m16_nkv8_n9216_consecutive", M=16, num_kv_heads=8, max_pos=32768,
              num_pages=4096, seed=1003, consecutive=True))
# token-count sweep with wide x and outlier rows
for _m in SWEEP_M:
    _add(Workload(f"sweep_m{_m}_nkv8_n9216", M=_m, num_kv_heads=8, max_pos=32768,
                  num_pages=4096, seed=1004 + _m, x_std=2.0, outlier_rows=True))
# sixteen KV heads: N = 18432, W ~302 MB
_add(Workload("m8_nkv16_n18432", M=8, num_kv_heads=16, max_pos=131072, num_pages=8192,
              seed=1005))

BENCH_WORKLOAD = "m8_nkv8_n9216"


def rope_table(max_pos: int, rot_dim: int = HEAD_DIM, base: float = ROPE_BASE) -> torch.Tensor:
    """fp32 [max_pos, rot_dim]: cos(pos * base^(-2i/rot_dim)) in columns i < rot_dim/2,
    the matching sin in columns rot_dim/2 + i (computed in float64, then rounded)."""
    half = rot_dim // 2
    inv_freq = base ** (-(np.arange(half, dtype=np.float64) * 2.0) / rot_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(table))


def _slots(w: Workload, g: torch.Generator) -> torch.Tensor:
    total = w.num_pages * PAGE_SLOTS
    if not w.consecutive:
        return torch.randperm(total, generator=g)[: w.M].to(torch.int64)
    # logical slots are consecutive; physically page P1 offsets o..15 then
    # page P2 offsets 0..o-1, with P2 not the page after P1
    while True:
        p1, p2 = (int(v) for v in torch.randint(0, w.num_pages, (2,), generator=g))
        if p1 != p2 and p2 != p1 + 1:
            break
    o = int(torch.randint(1, PAGE_SLOTS, (1,), generator=g))
    first = [p1 * PAGE_SLOTS + o + i for i in range(PAGE_SLOTS - o)]
    second = [p2 * PAGE_SLOTS + i for i in range(o)]
    return torch.tensor((first + second)[: w.M], dtype=torch.int64)


def make_inputs(w: Workload, integer_valued: bool = False) -> dict:
    """CPU tensors of one call: x, W (bf16), positions, slots (int64), cos_sin
    (fp32), kv_cache (bf16, pre-filled N(0,1)).

    ``integer_valued`` draws x and W from {-4..4} instead, which makes every
    FP32 partial sum of the projection exact in any order.
    """
    g = torch.Generator().manual_seed(w.seed)
    M, N = w.M, w.N
    if integer_valued:
        x = torch.randint(-4, 5, (M, HIDDEN), generator=g).to(torch.bfloat16)
        W = torch.randint(-4, 5, (N, HIDDEN), generator=g).to(torch.bfloat16)
    else:
        x = torch.randn(M, HIDDEN, generator=g) * w.x_std
        if w.outlier_rows:
            hit = torch.rand(M, generator=g) < 0.01
            if M >= 4 and not bool(hit.any()):
                hit[int(torch.randint(0, M, (1,), generator=g))] = True
            x[hit] *= 100.0
        x = x.to(torch.bfloat16)
        W = (torch.randn(N, HIDDEN, generator=g) * (1.0 / math.sqrt(HIDDEN))).to(torch.bfloat16)
    if w.consecutive:
        p0 = int(torch.randint(0, w.max_pos - M + 1, (1,), generator=g))
        positions = torch.arange(p0, p0 + M, dtype=torch.int64)
    else:
        positions = torch.randint(0, w.max_pos, (M,), generator=g, dtype=torch.int64)
    slots = _slots(w, g)
    cos_sin = rope_table(w.max_pos)
    kv_cache = torch.randn(w.num_pages, w.num_kv_heads, PAGE_SLOTS, SLOT_WIDTH,
                           generator=g).to(torch.bfloat16)
    return {"x": x, "W": W, "positions": positions, "slots": slots, "cos_sin": cos_sin,
            "kv_cache": kv_cache}


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a CPU bf16 tensor (a view, no conversion)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("bf16 tensor expected")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """CPU bf16 tensor with the given uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


# ---- the standalone epilogue (unfused path; any number of tokens) -----------

@dataclasses.dataclass(frozen=True)
class EpiWorkload:
    """Tokens of one prefill chunk: a BF16 projection output qkv [T, N] to be
    normed, rotated and inserted; positions p0..p0+T-1 and consecutive slots
    starting at a random page (one request's pages, in order)."""
    name: str
    T: int
    num_kv_heads: int
    max_pos: int
    num_pages: int
    seed: int
    qkv_std: float = 1.0

    @property
    def N(self) -> int:
        return columns_for(self.num_kv_heads)

    def roofline_bytes(self) -> int:
        """Algorithmic HBM bytes of one call: q/k/v heads read, q/k heads and
        K/V slot halves written, a table row and two indices per token."""
        head = HEAD_DIM * 2
        per_token = (9 + 1 + 9 + 2) * self.num_kv_heads * head + HEAD_DIM * 4 + 16
        return self.T * per_token

    def describe(self) -> dict:
        return {"workload": self.name, "T": self.T, "N": self.N, "num_kv_heads": self.num_kv_heads,
                "head_dim": HEAD_DIM, "cos_sin_rows": self.max_pos, "cache_pages": self.num_pages}


EPI_WORKLOADS: dict[str, EpiWorkload] = {}
for _w in (EpiWorkload("epi_t17_nkv1", T=17, num_kv_heads=1, max_pos=4096, num_pages=16, seed=3001),
           EpiWorkload("epi_t1000_nkv8", T=1000, num_kv_heads=8, max_pos=32768, num_pages=1024,
                       seed=3002, qkv_std=3.0),
           EpiWorkload("prefill_t4096_nkv8", T=4096, num_kv_heads=8, max_pos=32768, num_pages=4096,
                       seed=3003),
           EpiWorkload("prefill_t8192_nkv16", T=8192, num_kv_heads=16, max_pos=131072,
                       num_pages=8192, seed=3004)):
    EPI_WORKLOADS[_w.name] = _w

EPI_BENCH_WORKLOAD = "prefill_t4096_nkv8"


def make_epi_inputs(w: EpiWorkload) -> dict:
    """CPU tensors: qkv (bf16 [T, N], N(0, qkv_std^2)), positions, slots (int64),
    cos_sin (fp32), kv_cache (bf16, pre-filled N(0, 1))."""
    g = torch.Generator().manual_seed(w.seed)
    qkv = (torch.randn(w.T, w.N, generator=g) * w.qkv_std).to(torch.bfloat16)
    p0 = int(torch.randint(0, w.max_pos - w.T + 1, (1,), generator=g))
    positions = torch.arange(p0, p0 + w.T, dtype=torch.int64)
    pages_needed = (w.T + PAGE_SLOTS - 1) // PAGE_SLOTS + 1
    first_page = int(torch.randint(0, w.num_pages - pages_needed + 1, (1,), generator=g))
    o = int(torch.randint(0, PAGE_SLOTS, (1,), generator=g))
    slots = torch.arange(first_page * PAGE_SLOTS + o, first_page * PAGE_SLOTS + o + w.T,
                         dtype=torch.int64)
    cos_sin = rope_table(w.max_pos)
    kv_cache = torch.randn(w.num_pages, w.num_kv_heads, PAGE_SLOTS, SLOT_WIDTH,
                           generator=g).to(torch.bfloat16)
    return {"qkv": qkv, "positions": positions, "slots": slots, "cos_sin": cos_sin,
            "kv_cache": kv_cache}


# ---- the predecessor of the front (first layer's front) ---------------------

def make_layer_front_inputs(w: Workload) -> dict:
    """Embedded tokens x_embed (bf16 [M, 8192], N(0, 1)) and the pre-QKV norm
    weight (bf16 [8192], 1 + N(0, 0.1^2)), seeded from the workload's seed."""
    g = torch.Generator().manual_seed(w.seed + 7919)
    x_embed = torch.randn(w.M, HIDDEN, generator=g).to(torch.bfloat16)
    weight = (1.0 + 0.1 * torch.randn(HIDDEN, generator=g)).to(torch.bfloat16)
    return {"x_embed": x_embed, "norm_weight": weight}


# ---- the cache's consumer: verify-step paged attention (attn2) --------------

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """R requests of the 8-token verify step (rows 8r..8r+7 of qkv), each with
    its context length and its pages scattered over the cache."""
    name: str
    R: int
    num_kv_heads: int
    context: tuple          # one length per request (>= 8)
    num_pages: int
    seed: int
    window: int = 0

    @property
    def N(self) -> int:
        return columns_for(self.num_kv_heads)

    def max_blocks(self) -> int:
        return max((L + PAGE_SLOTS - 1) // PAGE_SLOTS for L in self.context)

    def roofline_bytes(self) -> int:
        """Algorithmic HBM bytes of one call: the K | V slots each request's
        rows can see (read once per KV head), the q and gate heads read, the
        output written, the block table and lengths."""
        kv = 0
        for L in self.context:
            lo = max(0, L - 8 - self.window + 1) if self.window else 0
            kv += (L - lo) * self.num_kv_heads * SLOT_WIDTH * 2
        q_gate = self.R * 8 * 2 * Q_PER_KV * self.num_kv_heads * HEAD_DIM * 2
        out = self.R * 8 * Q_PER_KV * self.num_kv_heads * HEAD_DIM * 2
        return kv + q_gate + out + self.R * (self.max_blocks() * 4 + 4)

    def describe(self) -> dict:
        return {"workload": self.name, "requests": self.R, "query_rows": 8 * self.R,
                "num_kv_heads": self.num_kv_heads, "context": list(self.context),
                "window": self.window, "cache_pages": self.num_pages}


ATTN_WORKLOADS: dict[str, AttnWorkload] = {}
for _a in (AttnWorkload("attn_r1_l8_nkv1", R=1, num_kv_heads=1, context=(8,), num_pages=4, seed=5001),
           AttnWorkload("attn_r3_mixed_nkv2", R=3, num_kv_heads=2, context=(8, 37, 300),
                        num_pages=64, seed=5002),
           AttnWorkload("attn_r2_window_nkv8", R=2, num_kv_heads=8, context=(700, 2051),
                        num_pages=512, seed=5003, window=128),
           AttnWorkload("attn_r1_l32k_nkv8", R=1, num_kv_heads=8, context=(32768,), num_pages=4096,
                        seed=5004),
           AttnWorkload("attn_r8_l4k_nkv8", R=8, num_kv_heads=8, context=(4096,) * 8,
                        num_pages=4096, seed=5005),
           AttnWorkload("attn_r32_l1k_nkv8", R=32, num_kv_heads=8, context=(1024,) * 32,
                        num_pages=4096, seed=5006)):
    ATTN_WORKLOADS[_a.name] = _a

ATTN_BENCH_WORKLOAD = "attn_r1_l32k_nkv8"


def make_attn_inputs(w: AttnWorkload) -> dict:
    """qkv (bf16 [8R, N], N(0, 1): q heads, gate heads and the rest), the
    cache (bf16, N(0, 1)), a block table (int32 [R, max_blocks]) giving each
    request distinct pages in random order, context lengths (int32 [R])."""
    g = torch.Generator().manual_seed(w.seed)
    qkv = torch.randn(8 * w.R, w.N, generator=g).to(torch.bfloat16)
    kv_cache = torch.randn(w.num_pages, w.num_kv_heads, PAGE_SLOTS, SLOT_WIDTH,
                           generator=g).to(torch.bfloat16)
    mb = w.max_blocks()
    need = sum((L + PAGE_SLOTS - 1) // PAGE_SLOTS for L in w.context)
    if need > w.num_pages:
        raise ValueError("not enough cache pages for the contexts")
    perm = torch.randperm(w.num_pages, generator=g)[:need]
    table = torch.full((w.R, mb), -1, dtype=torch.int32)
    k = 0
    for r, L in enumerate(w.context):
        nb = (L + PAGE_SLOTS - 1) // PAGE_SLOTS
        table[r, :nb] = perm[k:k + nb].to(torch.int32)
        k += nb
    lens = torch.tensor(w.context, dtype=torch.int32)
    return {"qkv": qkv, "kv_cache": kv_cache, "block_table": table, "context_lens": lens}
