"""Seeded synthetic inputs for the compressed-KV decode path.

This module holds the input recipes only: it draws keys, values and queries
and does none of the method's arithmetic (no basis, no selection, no packing,
no attention).  The oracle side and the CUDA side both take their inputs from
here, so they see identical bytes.

Shapes follow a Llama-3.1-8B-style attention layer (8 KV heads, 32 query heads,
head dim 128), the model the MosaicKV paper (arXiv 2607.00760, §1 Introduction
and §2.1) uses for its KV-size arithmetic.  The paper's LongBench and RULER
data and model weights are not available; these generators stand in for them.

Recipe for one (layer, batch b, KV head h) stream of K (V is the same with its
own decay and its own rotation):

    X = (Z * M) @ diag(sigma) @ Q_h            then rounded to fp16 (RNE)

    Z ~ N(0, 1) of shape [T, 128]
    M = `mult` with probability `p_out`, else 1   (elementwise outliers)
    sigma_i = exp(-i / decay)                      (spectral decay)
    Q_h = Haar-random orthogonal (QR of a Gaussian, sign of diag(R) fixed),
          drawn per (layer, KV head) and shared by every batch entry.

Queries: query head i belongs to KV head i // g (g = Hq / H).  Each query is
a uniformly chosen cached key of its KV head plus N(0, 0.5^2) noise, rounded
to fp16.

The mixed-regime workload assigns each compression segment one of three regimes
by segment index mod 3: near-low-rank (decay 8), flat (sigma_i = 1) and
outlier-heavy (base decay, 10% outliers x16).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_kv_heads: int
    n_q_heads: int
    ctx: int
    segment: int
    c: int
    tau: float
    top_k: int
    seed: int
    layers: int = 1
    decay_k: float = 24.0
    decay_v: float = 48.0
    # per-layer decay drawn uniformly from this range (K); V uses twice it
    decay_range: Optional[tuple] = None
    mixed_regimes: bool = False
    p_out: float = 0.02
    mult: float = 8.0
    q_noise: float = 0.5

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def streams(self) -> int:
        return self.batch * self.n_kv_heads


# The five workloads: a tiny correctness case, a 32K-context layer, the 128K
# batch-8 headline layer (32 layers), a 1M-token single sequence (32 layers),
# and a mixed-strategy 256K-context stress case.
TINY_4K = Workload("tiny-4K-b1", 1, 8, 32, 4096, 64, 64, 0.9, 256, seed=0)
LAYER_32K = Workload("llama8b-32K-b4", 4, 8, 32, 32768, 64, 40, 0.85, 2048, seed=1)
HEADLINE_128K = Workload("llama8b-128K-b8-x32", 8, 8, 32, 131072, 128, 40, 0.85, 4096,
                         seed=2, layers=32, decay_range=(16.0, 40.0))
MILLION_1M = Workload("llama8b-1M-b1-x32", 1, 8, 32, 1048576, 128, 32, 0.8, 8192,
                      seed=3, layers=32)
MIXED_256K = Workload("mixed-256K-b4-g7", 4, 4, 28, 262144, 64, 48, 0.9, 4096,
                      seed=4, mixed_regimes=True)

WORKLOADS = {w.name: w for w in (TINY_4K, LAYER_32K, HEADLINE_128K, MILLION_1M, MIXED_256K)}


def _gen(seed: int, layer: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + layer * 10_007 + tag * 101) & 0x7FFF_FFFF_FFFF)
    return g


def haar_orthogonal(n_mats: int, gen: torch.Generator, device=None) -> torch.Tensor:
    """[n_mats, 128, 128] fp32 Haar-random orthogonal matrices, drawn and
    factored on the CPU (`gen` is a CPU generator), returned on `device`."""
    a = torch.randn(n_mats, HEAD_DIM, HEAD_DIM, generator=gen, dtype=torch.float64)
    q, r = torch.linalg.qr(a)
    s = torch.sign(torch.diagonal(r, dim1=-2, dim2=-1))
    s[s == 0] = 1.0
    out = (q * s.unsqueeze(-2)).to(torch.float32)
    return out if device is None else out.to(device)


def layer_decays(w: Workload, layer: int):
    """(decay_K, decay_V) for a layer."""
    if w.decay_range is None:
        return w.decay_k, w.decay_v
    g = _gen(w.seed, layer, 7, "cpu")
    lo, hi = w.decay_range
    dk = lo + (hi - lo) * float(torch.rand(1, generator=g, dtype=torch.float64))
    return dk, 2.0 * dk


def _sigma(decay: float, device) -> torch.Tensor:
    i = torch.arange(HEAD_DIM, device=device, dtype=torch.float32)
    return torch.exp(-i / decay)


def _draw(w: Workload, layer: int, which: int, decay: float, device,
          ctx: Optional[int] = None, streams: Optional[int] = None) -> torch.Tensor:
    """One of K (which=0) or V (which=1): fp16 [B, H, T, 128] on `device`.
    streams=1 draws a single stream [1, 1, T, 128] with the same recipe (its
    own random values)."""
    T = w.ctx if ctx is None else ctx
    B, H = w.batch, w.n_kv_heads
    gen = _gen(w.seed, layer, 1 + which, device)
    Q = haar_orthogonal(H, _gen(w.seed, layer, 11 + which, "cpu"), device)   # [H, 128, 128]
    if streams == 1:
        B, H = 1, 1
    out = torch.empty(B, H, T, HEAD_DIM, dtype=torch.float16, device=device)
    if w.mixed_regimes:
        regime = (torch.arange(T, device=device) // w.segment) % 3     # [T]
        sig_tab = torch.stack([_sigma(8.0, device), torch.ones(HEAD_DIM, device=device),
                               _sigma(decay, device)])                 # [3, 128]
        sig = sig_tab[regime]                                          # [T, 128]
        heavy = (regime == 2).view(T, 1)
        p_out = torch.where(heavy, 0.10, w.p_out)                      # [T, 1]
        mult = torch.where(heavy, 16.0, w.mult)                        # [T, 1]
    else:
        sig = _sigma(decay, device).view(1, HEAD_DIM)
        p_out = torch.full((1, 1), w.p_out, device=device)
        mult = torch.full((1, 1), w.mult, device=device)
    # one batch entry (all H heads) per draw keeps the scratch at [H, T, 128]
    for b in range(B):
        z = torch.randn(H, T, HEAD_DIM, generator=gen, device=device)
        u = torch.rand(H, T, HEAD_DIM, generator=gen, device=device)
        m = torch.where(u < p_out, mult, 1.0)
        out[b] = torch.bmm(z * m * sig, Q[:H]).to(torch.float16)
        del z, u, m
    return out


def draw_kv(w: Workload, layer: int = 0, device="cpu", ctx: Optional[int] = None,
            streams: Optional[int] = None):
    """(K, V) fp16 [B, H, T, 128] for one layer."""
    dk, dv = layer_decays(w, layer)
    return (_draw(w, layer, 0, dk, device, ctx, streams),
            _draw(w, layer, 1, dv, device, ctx, streams))


def draw_queries(w: Workload, K: torch.Tensor, layer: int = 0, step: int = 0) -> torch.Tensor:
    """fp16 [B, Hq, 128]: a random cached key of the head plus N(0, 0.5^2) noise."""
    B, H, T, D = K.shape
    g = w.n_q_heads // H
    dev = K.device
    gen = _gen(w.seed, layer, 50 + step, dev)
    t_idx = torch.randint(0, T, (B, w.n_q_heads), generator=gen, device=dev)
    head = torch.arange(w.n_q_heads, device=dev) // g
    base = K[torch.arange(B, device=dev).view(B, 1), head.view(1, -1), t_idx]   # [B, Hq, D]
    noise = torch.randn(B, w.n_q_heads, D, generator=gen, device=dev) * w.q_noise
    return (base.float() + noise).to(torch.float16)


def kv_cache_bytes(batch: int, ctx: int, layers: int, n_kv_heads: int,
                   head_dim: int = HEAD_DIM, elem_bytes: int = 2) -> int:
    """Uncompressed K+V bytes for a model shape."""
    return batch * ctx * layers * n_kv_heads * head_dim * 2 * elem_bytes


def small_workload(name: str, **kw) -> Workload:
    """A derived workload for edge-case tests (ragged tails, tiny k, ...)."""
    base = dict(name=name, batch=1, n_kv_heads=2, n_q_heads=4, ctx=300, segment=64,
                c=40, tau=0.85, top_k=32, seed=11)
    base.update(kw)
    return Workload(**base)

