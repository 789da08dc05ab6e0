"""Seeded synthetic inputs for the MLA latent pre-projection workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no normalization, no quantization), so both the CUDA path
and the CPU oracle can take their inputs from it.  Everything is generated on
the CPU with torch.Generator and returned as CPU tensors; callers copy the same
bits to the GPU.

Shapes follow DeepSeek-V4 MLA: q-lora rank 1536, kv latent 512, 64 rope
columns after them in the fused projection output (PR #53540 prhub summary,
attention.py snippet: qr_kv.split([q_lora_rank, head_dim], -1)), attention
wq_b N=24576 and indexer wq_b N=4096 over K=1536.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

KQ = 1536          # q-lora rank
KKV = 512          # kv latent width
ROPE = 64          # trailing rope columns of the fused projection row
ROW = KQ + KKV + ROPE
N_ATTN = 24576     # attention wq_b output features
N_IDX = 4096       # indexer wq_b output features
EPS = 1e-6


def _gen(seed: int, salt: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 1_000_003 + salt)
    return g


def gammas(seed: int, kq: int = KQ, kkv: int = KKV):
    """gamma_q, gamma_kv: bf16 U(0.5, 1.5)."""
    g = _gen(seed, 7)
    gq = (torch.rand(kq, generator=g) + 0.5).to(torch.bfloat16)
    gkv = (torch.rand(kkv, generator=g) + 0.5).to(torch.bfloat16)
    return gq, gkv


def student_t(shape, df: int, g: torch.Generator) -> torch.Tensor:
    """Student-t(df) draws by their definition z / sqrt(chi2_df / df), with
    chi2_df a sum of df squared standard normals."""
    z = torch.randn(shape, generator=g)
    chi2 = torch.zeros(shape)
    for _ in range(df):
        chi2 += torch.randn(shape, generator=g) ** 2
    return z / torch.sqrt(chi2 / df)


@dataclass
class Latents:
    """One batch of token rows.  When `buf` is set, q and kv are strided split
    views of it (row stride ROW); otherwise they are contiguous."""
    q: torch.Tensor          # bf16 [M, KQ] (possibly a view)
    kv: torch.Tensor         # bf16 [M, KKV] (possibly a view)
    gamma_q: torch.Tensor    # bf16 [KQ]
    gamma_kv: torch.Tensor   # bf16 [KKV]
    eps: float = EPS
    buf: torch.Tensor | None = None


def pr1_ref(seed: int = 0) -> Latents:
    """M=4 tokens, q [4,1536] and kv [4,512] N(0,1), gamma U(0.5,1.5)."""
    g = _gen(seed, 1)
    q = torch.randn(4, KQ, generator=g).to(torch.bfloat16)
    kv = torch.randn(4, KKV, generator=g).to(torch.bfloat16)
    gq, gkv = gammas(seed)
    return Latents(q, kv, gq, gkv)


def outlier_columns(seed: int, frac: float = 0.01, width: int = KQ + KKV) -> torch.Tensor:
    """ceil(frac * width) distinct column indices across q and kv."""
    n = math.ceil(frac * width)
    return torch.randperm(width, generator=_gen(seed, 3))[:n]


def decode_batch(M: int, seed: int = 1) -> Latents:
    """Decode sweep: one bf16 buffer [M, 2112] (q = cols 0:1536, kv =
    1536:2048, 64 unused rope columns), N(0,1) with 1% outlier channels x50."""
    g = _gen(seed, 100 + M)
    x = torch.randn(M, ROW, generator=g)
    cols = outlier_columns(seed)
    x[:, cols] *= 50.0
    buf = x.to(torch.bfloat16)
    gq, gkv = gammas(seed)
    return Latents(buf[:, :KQ], buf[:, KQ:KQ + KKV], gq, gkv, buf=buf)


def prefill_batch(M: int = 8192, seed: int = 2) -> Latents:
    """Prefill: contiguous q [M,1536] and kv [M,512], Student-t(df=4)."""
    g = _gen(seed, 200 + M)
    q = student_t((M, KQ), 4, g).to(torch.bfloat16)
    kv = student_t((M, KKV), 4, g).to(torch.bfloat16)
    gq, gkv = gammas(seed)
    return Latents(q, kv, gq, gkv)


def full_path_batch(M: int, seed: int = 3) -> Latents:
    """Full path: contiguous q [M,1536] and kv [M,512], N(0,1)."""
    g = _gen(seed, 300 + M)
    q = torch.randn(M, KQ, generator=g).to(torch.bfloat16)
    kv = torch.randn(M, KKV, generator=g).to(torch.bfloat16)
    gq, gkv = gammas(seed)
    return Latents(q, kv, gq, gkv)


def long_context_batch(M: int = 32768, seed: int = 4) -> Latents:
    """Long-context stress: N(0,1) plus edge rows.  Every 97th row has one
    all-zero q group (group index row mod 12); every 89th row has one
    single-spike q group (one element 1e3, the rest 0, group (row+5) mod 12,
    position row mod 128); rows 0 and M-1 are all zero (q and kv)."""
    g = _gen(seed, 400 + M)
    q = torch.randn(M, KQ, generator=g)
    kv = torch.randn(M, KKV, generator=g)
    G = KQ // 128
    for r in range(0, M, 97):
        gi = r % G
        q[r, gi * 128:(gi + 1) * 128] = 0.0
    for r in range(0, M, 89):
        gi = (r + 5) % G
        q[r, gi * 128:(gi + 1) * 128] = 0.0
        q[r, gi * 128 + r % 128] = 1e3
    for r in {0, M - 1}:
        q[r] = 0.0
        kv[r] = 0.0
    gq, gkv = gammas(seed)
    return Latents(q.to(torch.bfloat16), kv.to(torch.bfloat16), gq, gkv)


def weight(N: int, K: int = KQ, seed: int = 0, salt: int = 0, std: float = 0.02) -> torch.Tensor:
    """A wq_b weight [N, K] in fp32, N(0, std)."""
    g = _gen(seed, 900 + salt)
    return torch.randn(N, K, generator=g) * std


def activations_bf16(M: int, K: int, seed: int, zero_rows=()) -> torch.Tensor:
    """bf16 activations [M, K] N(0, 1) with 1% of the columns scaled by 30
    (outlier channels), and the listed rows all zero."""
    g = _gen(seed, 700 + M)
    x = torch.randn(M, K, generator=g)
    cols = torch.randperm(K, generator=g)[: max(1, K // 100)]
    x[:, cols] *= 30.0
    for r in zero_rows:
        x[r] = 0.0
    return x.to(torch.bfloat16)


def random_codes_and_scales(M: int, K: int, seed: int):
    """Arbitrary finite E4M3FN codes [M, K] (uint8, NaN codes excluded) and
    positive fp32 scales [M, K/128] drawn directly, for GEMM tests that need
    an A operand independent of any quantizer."""
    g = _gen(seed, 500 + M)
    codes = torch.randint(0, 256, (M, K), generator=g, dtype=torch.int32)
    codes = torch.where((codes & 0x7F) == 0x7F, codes - 1, codes).to(torch.uint8)
    scales = (torch.rand(M, K // 128, generator=g) * 0.02 + 0.001).float()
    return codes, scales


def bits(t: torch.Tensor):
    """uint16 numpy bit patterns of a bf16 CPU tensor (contiguous copy)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
