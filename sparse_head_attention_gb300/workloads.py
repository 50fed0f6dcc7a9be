"""Seeded synthetic workloads for the hybrid-head attention path.

This module only draws random inputs and names shapes; it holds none of the
method's arithmetic.  The tests hand the same tensors to the CUDA library and to
the fp64 oracle; the benchmark draws the same recipes on the device.

The shapes follow the pages' workloads: Llama-3.1-8B and Qwen3-8B attention
(32 query heads, 8 KV heads, head dim 128), contexts up to 256K as in RULER,
SSA sink/local sizes from the hyper-parameter table (128 / 2048), and the
XA-SSA setting (block-sparse retrieval heads plus streaming heads).  No dataset
or checkpoint is used: every tensor is N(0, 1) (router weights N(0, 0.02)).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import torch

FULL, SSA, BLOCK = 0, 1, 2
TILE = 128


@dataclass
class PrefillConfig:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    d: int
    sink: int
    window: int
    layers: int = 1
    # KV heads routed to SA (r = 1) in every batch element; None = router decides
    sa_heads: Optional[List[int]] = None
    fa_impl: int = FULL      # how an r = 0 head executes (FULL, or BLOCK for XA-SSA)
    sa_impl: int = SSA
    block_density: float = 0.2
    seed: int = 0


@dataclass
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int
    sink: int
    window: int
    sa_heads: List[int] = field(default_factory=list)
    seed: int = 0


def sa_heads_randperm(Hkv: int, n_sa: int, seed: int = 0) -> List[int]:
    """The seeded choice of SA heads: the first n_sa entries of randperm(Hkv)."""
    g = torch.Generator().manual_seed(seed)
    return sorted(torch.randperm(Hkv, generator=g)[:n_sa].tolist())


TINY = PrefillConfig("tiny_prefill_s1k_fa_ssa", B=1, S=1024, Hq=8, Hkv=2, d=128,
                     sink=64, window=256, sa_heads=[1])
LLAMA_32K = PrefillConfig("llama3_8b_layer_prefill_s32k_fa_ssa", B=1, S=32768, Hq=32, Hkv=8,
                          d=128, sink=128, window=2048, sa_heads=sa_heads_randperm(8, 6, 0))
QWEN_64K_36L = PrefillConfig("qwen3_8b_36layer_prefill_s64k_routed", B=1, S=65536, Hq=32,
                             Hkv=8, d=128, sink=128, window=2048, layers=36, sa_heads=None)
XA_SSA_256K = PrefillConfig("xa_ssa_prefill_s256k", B=1, S=262144, Hq=32, Hkv=8, d=128,
                            sink=128, window=4096, sa_heads=sa_heads_randperm(8, 6, 0),
                            fa_impl=BLOCK, sa_impl=SSA)
DECODE_128K = DecodeConfig("decode_b32_l128k_fa_ssa", B=32, Hq=32, Hkv=8, d=128, L=131072,
                           sink=128, window=4096, sa_heads=sa_heads_randperm(8, 6, 0))

PREFILL_CONFIGS = {c.name: c for c in (TINY, LLAMA_32K, QWEN_64K_36L, XA_SSA_256K)}
DECODE_CONFIGS = {DECODE_128K.name: DECODE_128K}


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in float32 with a seeded generator, rounded to bf16."""
    return torch.randn(shape, generator=_gen(seed, device), device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def qkv(B, S, Hq, Hkv, d, seed=0, device="cpu"):
    """Q [B, S, Hq, d], K and V [B, S, Hkv, d], bf16 N(0, 1), seeds seed*3 + {0,1,2}."""
    Q = randn_bf16((B, S, Hq, d), 3 * seed + 0, device)
    K = randn_bf16((B, S, Hkv, d), 3 * seed + 1, device)
    V = randn_bf16((B, S, Hkv, d), 3 * seed + 2, device)
    return Q, K, V


def offset_values(B, S, Hkv, d, seed=0, lo=2.2, hi=3.8, device="cpu"):
    """V [B, S, Hkv, d] bf16 with |v| uniform in [lo, hi) and one sign per
    (b, KV head, dim) for all positions: any convex combination of a head's
    values then has |O| in [lo, hi) too (a stress input for the output's
    absolute error, which grows with |O|)."""
    g = _gen(seed, device)
    mag = lo + (hi - lo) * torch.rand((B, S, Hkv, d), generator=g, device=device)
    sign = torch.where(torch.rand((B, 1, Hkv, d), generator=g, device=device) < 0.5, -1.0, 1.0)
    return (mag * sign).to(torch.bfloat16)


def routing_from_sa_heads(B: int, Hkv: int, sa_heads, fa_impl=FULL, sa_impl=SSA):
    """(r, m) uint8 [B, Hkv] for a fixed set of SA heads (same in every batch row)."""
    r = torch.zeros((B, Hkv), dtype=torch.uint8)
    for h in sa_heads:
        r[:, h] = 1
    m = torch.where(r == 1, torch.tensor(sa_impl, dtype=torch.uint8),
                    torch.tensor(fa_impl, dtype=torch.uint8))
    return r, m


def block_mask(B: int, Hkv: int, S: int, density: float = 0.2, seed: int = 0,
               T: int = TILE) -> torch.Tensor:
    """uint8 [B, Hkv, nB, nB] causal block mask: the diagonal block and key block 0
    are always kept; every other block below the diagonal is kept with
    probability `density` (uniforms drawn in (b, h, qb, kb) order); blocks above
    the diagonal are 0."""
    nB = (S + T - 1) // T
    u = torch.rand((B, Hkv, nB, nB), generator=_gen(seed, "cpu"))
    keep = u < density
    idx = torch.arange(nB)
    lower = idx[None, :] <= idx[:, None]          # kb <= qb
    keep = keep & lower
    keep[..., idx, idx] = True                     # diagonal
    keep[..., :, 0] = True                         # first key block
    return keep.to(torch.uint8)


def xa_planted_qk(B: int, S: int, Hq: int, Hkv: int, d: int, hot_frac: float = 0.05,
                  gain: float = 0.67, seed: int = 0, device="cpu"):
    """Q [B, S, Hq, d] and K [B, S, Hkv, d] bf16 with planted block structure, for
    block-mask estimation: N(0, 1) entries (seeds 3*seed + {0, 1}); then, per
    (b, KV head), a vector v of entries +-gain (random signs) is added to every
    query of the heads that read it and to every key of a random set of 128-token
    "hot" key blocks (each block hot with probability hot_frac; key block 0 always
    hot).  Values are drawn in float32 and rounded to bf16 once, at the end."""
    g = Hq // Hkv
    Q = torch.randn((B, S, Hq, d), generator=_gen(3 * seed + 0, device), device=device)
    K = torch.randn((B, S, Hkv, d), generator=_gen(3 * seed + 1, device), device=device)
    nB = (S + TILE - 1) // TILE
    gc = _gen(7919 * seed + 17, "cpu")
    for b in range(B):
        for h in range(Hkv):
            v = (torch.randint(0, 2, (d,), generator=gc).float() * 2 - 1) * gain
            hot = torch.rand(nB, generator=gc) < hot_frac
            hot[0] = True
            v = v.to(device)
            Q[b, :, h * g:(h + 1) * g, :] += v
            tok_hot = hot.repeat_interleave(TILE)[:S].to(device)
            K[b, tok_hot, h, :] += v
    return Q.to(torch.bfloat16), K.to(torch.bfloat16)


def router_weights(layer: int, d: int = 128, hidden: int = 64, seed: int = 0,
                   beta: float = 0.0, device="cpu"):
    """Weights of the 2-layer router MLP d -> hidden -> 2 for one layer:
    W ~ N(0, 0.02) (seed + layer), hidden bias 0, output bias [0, beta]."""
    g = _gen(seed + layer, "cpu")
    W1 = (torch.randn((hidden, d), generator=g) * 0.02).float()
    W2 = (torch.randn((2, hidden), generator=g) * 0.02).float()
    b1 = torch.zeros(hidden, dtype=torch.float32)
    b2 = torch.tensor([0.0, beta], dtype=torch.float32)
    return [W1.to(device), W2.to(device)], [b1.to(device), b2.to(device)]


def decode_inputs(cfg: DecodeConfig, device="cpu", Lmax: Optional[int] = None, seqlens=None):
    """q [B, Hq, d], K/V cache [B, Lmax, Hkv, d] (bf16 N(0, 1)), seqlens int32 [B]."""
    Lmax = Lmax or cfg.L
    s = 3 * cfg.seed + 100
    q = randn_bf16((cfg.B, cfg.Hq, cfg.d), s, device)
    Kc = randn_bf16((cfg.B, Lmax, cfg.Hkv, cfg.d), s + 1, device)
    Vc = randn_bf16((cfg.B, Lmax, cfg.Hkv, cfg.d), s + 2, device)
    if seqlens is None:
        seqlens = torch.full((cfg.B,), cfg.L, dtype=torch.int32)
    return q, Kc, Vc, torch.as_tensor(seqlens, dtype=torch.int32).to(device)
